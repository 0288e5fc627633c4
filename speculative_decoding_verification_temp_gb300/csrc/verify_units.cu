// Fused chain/tree verification kernel and the residual-output kernel.
// See verify_units.cuh for the design.
#include <climits>

#include "verify_units.cuh"

namespace sv {

template <typename TE>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kKeyRounds = 4;
};
template <>
struct Elem<uint16_t> {
  static constexpr int kKeyRounds = 2;
};

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
// loading a vocabulary slice into shared memory
// ---------------------------------------------------------------------------

template <typename TE, bool kVec>
__device__ __forceinline__ void load_slice(TE *dst, const TE *src, int len) {
  if (kVec) {
    constexpr int kPer = 16 / sizeof(TE);
    const int nvec = len / kPer;
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src);
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
    int i = threadIdx.x;
    for (; i + 3 * kThreads < nvec; i += 4 * kThreads) {
      const uint4 a = __ldcs(s4 + i);
      const uint4 b = __ldcs(s4 + i + kThreads);
      const uint4 c = __ldcs(s4 + i + 2 * kThreads);
      const uint4 d = __ldcs(s4 + i + 3 * kThreads);
      d4[i] = a;
      d4[i + kThreads] = b;
      d4[i + 2 * kThreads] = c;
      d4[i + 3 * kThreads] = d;
    }
    for (; i < nvec; i += kThreads) d4[i] = __ldcs(s4 + i);
    for (int e = nvec * kPer + threadIdx.x; e < len; e += kThreads) dst[e] = src[e];
  } else {
    for (int e = threadIdx.x; e < len; e += kThreads) dst[e] = src[e];
  }
}

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
// per-CTA statistics of one slice
// ---------------------------------------------------------------------------

// Online max / sum of 2^((z - m) k) over the slice, optionally masked below
// the top-k threshold.  NaN shows up as a NaN sum (or flag bit 0 while the
// running max is still -inf), +inf as an infinite max.
template <typename TE>
__device__ void softmax_slice(const TE *s, int len, float k, float thr, bool masked, float &m,
                              float &S, int &fl) {
  m = -INFINITY;
  S = 0.f;
  fl = 0;
  float nmk = 0.f;
  for (int base = threadIdx.x * 8; base < len; base += kThreads * 8) {
    float z[8];
    load8<TE>(s, base, len, z);
    if (masked) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        if (z[e] != z[e]) fl |= 1;
        z[e] = z[e] >= thr ? z[e] : -INFINITY;
      }
    }
    float vm = fmaxf(fmaxf(fmaxf(z[0], z[1]), fmaxf(z[2], z[3])),
                     fmaxf(fmaxf(z[4], z[5]), fmaxf(z[6], z[7])));
    if (vm > m) {
      S *= fast_exp2((m - vm) * k);
      m = vm;
      nmk = -m * k;
    }
    if (m == -INFINITY) {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        if (z[e] != z[e]) fl |= 1;
      continue;
    }
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc += fast_exp2(fmaf(z[e], k, nmk));
    S += acc;
  }
}

// Argmax over the finite entries of the slice (lowest index on ties);
// flag bit 0: NaN seen, bit 1: +inf seen.
template <typename TE>
__device__ void argmax_slice(const TE *s, int len, int v0, float &bv, int &bi, int &fl) {
  bv = -INFINITY;
  bi = INT_MAX;
  fl = 0;
  for (int base = threadIdx.x * 8; base < len; base += kThreads * 8) {
    float z[8];
    load8<TE>(s, base, len, z);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float x = z[e];
      if (x != x) {
        fl |= 1;
      } else if (x == INFINITY) {
        fl |= 2;
      } else if (x > bv) {
        bv = x;
        bi = v0 + base + e;
      }
    }
  }
}

// Reduce a per-thread online (m, S, flags) triple over the CTA; the result is
// valid in every thread.
__device__ void block_online(float &m, float &S, int &fl, float k, Ctl &ctl) {
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
  __syncthreads();
  m = -INFINITY;
  S = 0.f;
  fl = 0;
  for (int w = 0; w < kWarps; ++w) {
    online_merge(m, S, ctl.red_f[0][w], ctl.red_f[1][w], k);
    fl |= ctl.red_i[0][w];
  }
  __syncthreads();
}

__device__ void block_argmax(float &bv, int &bi, int &fl, Ctl &ctl) {
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
  __syncthreads();
  bv = -INFINITY;
  bi = INT_MAX;
  fl = 0;
  for (int w = 0; w < kWarps; ++w) {
    argmax_merge(bv, bi, ctl.red_f[0][w], ctl.red_i[0][w]);
    fl |= ctl.red_i[1][w];
  }
  __syncthreads();
}

__device__ float block_sum(float v, Ctl &ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) ctl.red_f[0][warp] = v;
  __syncthreads();
  float r = 0.f;
  for (int w = 0; w < kWarps; ++w) r += ctl.red_f[0][w];
  __syncthreads();
  return r;
}

// ---------------------------------------------------------------------------
// cluster-wide top-k threshold: radix select on order keys, 8 bits per round
// ---------------------------------------------------------------------------

template <typename TE>
__device__ void topk_thresholds(const TE *sp, const TE *sq, int len, bool do_p, bool do_q,
                                int kp, int kq, Ctl &ctl, cg::cluster_group &cluster, int C,
                                float &thr_p, float &thr_q) {
  constexpr int R = Elem<TE>::kKeyRounds;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 2) {
    ctl.prefix[tid] = 0u;
    ctl.kk[tid] = tid == 0 ? kp : kq;
  }
  for (int round = 0; round < R; ++round) {
    const int buf = round & 1;
    const int shift = (R - 1 - round) * 8;
    for (int i = tid; i < 512; i += kThreads) (&ctl.hist[buf][0][0])[i] = 0;
    __syncthreads();
    const uint32_t hmask = static_cast<uint32_t>(~0ull << (shift + 8));
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (row == 0 ? !do_p : !do_q) continue;
      const TE *s = row == 0 ? sp : sq;
      const uint32_t want =
          static_cast<uint32_t>(static_cast<unsigned long long>(ctl.prefix[row]) << (shift + 8));
      for (int v = tid; v < len; v += kThreads) {
        const uint32_t key = order_key(s[v]);
        if ((key & hmask) == want) atomicAdd(&ctl.hist[buf][row][(key >> shift) & 255u], 1);
      }
    }
    __syncthreads();
    cluster.sync();
    for (int i = tid; i < 512; i += kThreads) {
      int g = 0;
      for (int r = 0; r < C; ++r) g += cluster.map_shared_rank(&ctl.hist[buf][0][0], r)[i];
      (&ctl.ghist[0][0])[i] = g;
    }
    __syncthreads();
    if (warp < 2 && (warp == 0 ? do_p : do_q)) {
      const int row = warp;
      int cnt[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = ctl.ghist[row][255 - 8 * lane - j];
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
    __syncthreads();
  }
  if (sizeof(TE) == 2) {
    thr_p = key_value_bf16(ctl.prefix[0]);
    thr_q = key_value_bf16(ctl.prefix[1]);
  } else {
    thr_p = key_value_f32(ctl.prefix[0]);
    thr_q = key_value_f32(ctl.prefix[1]);
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// inverse-CDF search inside the CTA that owns the threshold
// ---------------------------------------------------------------------------

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
    ctl.red_f[0][warp] = sum;
    ctl.red_i[0][warp] = lastpos;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float acc = 0.f;
    int owner = -1;
    float trel = INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      const float tw = ctl.red_f[0][w];
      if (acc + tw > t) {
        owner = w;
        trel = t - acc;
        break;
      }
      acc += tw;
    }
    if (owner < 0) {
      for (int w = kWarps - 1; w >= 0; --w)
        if (ctl.red_i[0][w] >= 0) {
          owner = w;
          break;
        }
      trel = INFINITY;
    }
    ctl.owner_warp = owner;
    ctl.owner_t = trel;
    ctl.token_local = -1;
  }
  __syncthreads();
  if (warp == ctl.owner_warp) {
    const float trel = ctl.owner_t;
    const int ocs = warp * L, oce = min(len, ocs + L);
    float base_sum = 0.f;
    int result = -1;
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
        if (lane == first) {
          float run = base_sum + excl;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            run += w[e];
            if (found < 0 && w[e] > 0.f && run > trel) found = base + e;
          }
          if (found < 0) found = lp;
        }
        result = __shfl_sync(0xFFFFFFFFu, found, first);
      }
      base_sum += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (result < 0) result = ctl.red_i[0][warp];
    if (lane == 0) ctl.token_local = v0 + result;
  }
  __syncthreads();
  const int tok = ctl.token_local;
  __syncthreads();
  return tok;
}

// ---------------------------------------------------------------------------
// the unit kernel
// ---------------------------------------------------------------------------

__device__ __forceinline__ const void *row_ptr(const void *base, long long row, long long ld,
                                               int esize) {
  return static_cast<const char *>(base) + (row * ld) * esize;
}

// Next child of `node` with id > after, or -1 (CTA-collective).
__device__ int next_child(const Params &P, int seq, int node, int after, Ctl &ctl) {
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
  __syncthreads();
  const int r = ctl.child;
  __syncthreads();
  return r;
}

__device__ __forceinline__ int child_token(const Params &P, int seq, int node, int child) {
  if (P.mode == kModeChain) return __ldg(P.tokens + static_cast<long long>(seq) * P.gamma + node);
  return __ldg(P.tokens + static_cast<long long>(seq) * P.ups + child);
}

__device__ __forceinline__ float unit_uniform(const Params &P, int seq, int pos, int draw) {
  if (P.uov) return __ldg(P.uov + (static_cast<long long>(seq) * P.ups + pos) * 2 + draw);
  return philox_uniform(P.seed, static_cast<uint32_t>(seq), static_cast<uint32_t>(pos),
                        static_cast<uint32_t>(draw));
}

template <typename TE>
__device__ __forceinline__ float gather_z(const TE *row_base, int x, int slice,
                                          cg::cluster_group &cluster) {
  const int r = x / slice;
  const TE *remote = cluster.map_shared_rank(row_base, r);
  return to_f32(remote[x - r * slice]);
}

// Sum of the current draw weights over the cluster; fills ctl.parts with the
// per-CTA totals in rank order.  Cluster-collective.
template <typename TE>
__device__ float cluster_total(const RowDesc &dp, const RowDesc &dq, int residual, float c,
                               const TE *sp, const TE *sq, int v0, int len, Ctl &ctl,
                               cg::cluster_group &cluster, int C, int &xround) {
  float acc = 0.f;
  for (int base = threadIdx.x * 8; base < len; base += kThreads * 8) {
    float zp[8], zq[8];
    load8<TE>(sp, base, len, zp);
    if (residual) load8<TE>(sq, base, len, zq);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (base + e < len)
        acc += weight(dp, dq, residual, c, zp[e], residual ? zq[e] : 0.f, v0 + base + e);
  }
  acc = block_sum(acc, ctl);
  const int buf = xround & 1;
  ++xround;
  if (threadIdx.x == 0) ctl.wx[buf][0] = acc;
  cluster.sync();
  float total = 0.f;
  for (int r = 0; r < C; ++r) {
    const float pr = cluster.map_shared_rank(&ctl.wx[buf][0], r)[0];
    if (threadIdx.x == 0) ctl.parts[r] = pr;
    total += pr;
  }
  __syncthreads();
  return total;
}

template <typename TE, bool kVec>
__global__ void __launch_bounds__(kThreads) unit_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Ctl &ctl = *reinterpret_cast<Ctl *>(smem_raw);
  TE *sp = reinterpret_cast<TE *>(smem_raw + P.ctl_bytes);
  TE *sq = sp + P.slice;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = P.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int unit = blockIdx.x / C;
  const int seq = unit / P.ups, node = unit % P.ups;
  const int tid = threadIdx.x;
  const int V = P.V;
  const int v0 = rank * P.slice;
  const int len = max(0, min(V, v0 + P.slice) - v0);

  const float Tp = __ldg(P.Tp + seq), Tq = __ldg(P.Tq + seq);
  const int kp_raw = P.kp ? __ldg(P.kp + seq) : 0;
  const int kq_raw = P.kq ? __ldg(P.kq + seq) : 0;
  const bool tp_bad = !(Tp >= 0.f) || Tp == INFINITY;
  const bool tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  const bool p_arg = tp_bad || Tp == 0.f;  // p decided by argmax
  const bool q_arg = tq_bad || Tq == 0.f;

  int child = next_child(P, seq, node, -1, ctl);
  const bool has_children = child >= 0;
  const bool load_q = has_children && !p_arg;

  long long prow, qrow;
  if (P.mode == kModeChain) {
    prow = static_cast<long long>(seq) * (P.gamma + 1) + node;
    qrow = static_cast<long long>(seq) * P.gamma + node;
  } else {
    prow = static_cast<long long>(seq) * P.ups + node;
    qrow = prow;
  }
  const TE *gp = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE))) + v0;
  load_slice<TE, kVec>(sp, gp, len);
  if (load_q) {
    const TE *gq = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE))) + v0;
    load_slice<TE, kVec>(sq, gq, len);
  }
  __syncthreads();

  // ---- top-k thresholds
  const bool topk_p = !p_arg && kp_raw > 0 && kp_raw < V;
  const bool topk_q = load_q && !q_arg && kq_raw > 0 && kq_raw < V;
  float thr_p = -INFINITY, thr_q = -INFINITY;
  if (topk_p || topk_q) {
    float tp, tq;
    topk_thresholds<TE>(sp, sq, len, topk_p, topk_q, kp_raw, kq_raw, ctl, cluster, C, tp, tq);
    if (topk_p) thr_p = tp;
    if (topk_q) thr_q = tq;
  }

  // ---- row statistics
  const float kpv = p_arg ? 0.f : kLog2e / Tp;
  const float kqv = q_arg ? 0.f : kLog2e / Tq;
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    if (row == 1 && !load_q) break;
    const TE *s = row == 0 ? sp : sq;
    const bool arg = row == 0 ? p_arg : q_arg;
    Partial pt;
    if (arg) {
      argmax_slice<TE>(s, len, v0, pt.av, pt.ai, pt.flags);
      block_argmax(pt.av, pt.ai, pt.flags, ctl);
      pt.m = 0.f;
      pt.S = 0.f;
    } else {
      const float kk = row == 0 ? kpv : kqv;
      const float thr = row == 0 ? thr_p : thr_q;
      const bool masked = row == 0 ? topk_p : topk_q;
      softmax_slice<TE>(s, len, kk, thr, masked, pt.m, pt.S, pt.flags);
      block_online(pt.m, pt.S, pt.flags, kk, ctl);
      pt.av = 0.f;
      pt.ai = 0;
    }
    if (tid == 0) ctl.part[row] = pt;
  }
  cluster.sync();

  RowDesc dp, dq;
  bool need_fallback[2] = {false, false};
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    RowDesc d;
    d.pad = 0;
    d.flags = 0u;
    d.thr = row == 0 ? thr_p : thr_q;
    const bool arg = row == 0 ? p_arg : q_arg;
    const bool tbad = row == 0 ? tp_bad : tq_bad;
    const float kk = row == 0 ? kpv : kqv;
    if (row == 1 && !load_q) {
      d.onehot = 1;
      d.a = 0;
      d.k = d.nmk = d.invS = 0.f;
      dq = d;
      break;
    }
    if (arg) {
      float bv = -INFINITY;
      int bi = INT_MAX, fl = 0;
      for (int r = 0; r < C; ++r) {
        const Partial o = cluster.map_shared_rank(&ctl.part[row], r)[0];
        argmax_merge(bv, bi, o.av, o.ai);
        fl |= o.flags;
      }
      d.onehot = 1;
      d.a = bi == INT_MAX ? 0 : bi;
      d.k = d.nmk = d.invS = 0.f;
      if (tbad || fl || bi == INT_MAX) d.flags = SPEC_FLAG_NONFINITE;
    } else {
      float M = -INFINITY, S = 0.f;
      int fl = 0;
      for (int r = 0; r < C; ++r) {
        const Partial o = cluster.map_shared_rank(&ctl.part[row], r)[0];
        online_merge(M, S, o.m, o.S, kk);
        fl |= o.flags;
      }
      const bool bad = fl || !(M > -INFINITY) || M == INFINITY || !(S > 0.f) || S == INFINITY ||
                       S != S;
      d.onehot = 0;
      d.a = 0;
      d.k = kk;
      d.nmk = -M * kk;
      d.invS = 1.f / S;
      if (bad) {
        need_fallback[row] = true;
        d.onehot = 1;
        d.flags = SPEC_FLAG_NONFINITE;
      }
    }
    if (row == 0) dp = d; else dq = d;
  }

  // ---- finite-argmax fallback for non-finite sampling rows (rare)
  if (need_fallback[0] || need_fallback[1]) {
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (!need_fallback[row]) continue;
      Partial pt;
      argmax_slice<TE>(row == 0 ? sp : sq, len, v0, pt.av, pt.ai, pt.flags);
      block_argmax(pt.av, pt.ai, pt.flags, ctl);
      if (tid == 0) ctl.amax[row] = pt;
    }
    cluster.sync();
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (!need_fallback[row]) continue;
      float bv = -INFINITY;
      int bi = INT_MAX;
      for (int r = 0; r < C; ++r) {
        const Partial o = cluster.map_shared_rank(&ctl.amax[row], r)[0];
        argmax_merge(bv, bi, o.av, o.ai);
      }
      if (row == 0) dp.a = bi == INT_MAX ? 0 : bi;
      else dq.a = bi == INT_MAX ? 0 : bi;
    }
  }

  // ---- local walk over the children
  uint32_t uflags = dp.flags;
  int next = -1, token = -1;
  int residual = 0;
  float c = 0.f, Wcur = 0.f;
  bool have_parts = false;
  int xround = 0;
  int kind = 0;
  float total = 0.f;
  if (dp.onehot) {
    for (; child >= 0; child = next_child(P, seq, node, child, ctl)) {
      const int x = child_token(P, seq, node, child);
      if (x < 0 || x >= V) uflags |= SPEC_FLAG_BAD_TOKEN;
      if (x == dp.a) {
        next = child;
        break;
      }
    }
    if (next < 0) {
      token = dp.a;
      kind = has_children ? 1 : 0;
    }
  } else {
    if (child >= 0) uflags |= dq.flags;
    for (; child >= 0; child = next_child(P, seq, node, child, ctl)) {
      const int x = child_token(P, seq, node, child);
      const int keypos = P.mode == kModeChain ? node : child;
      const float u = unit_uniform(P, seq, keypos, 0);
      bool acc = false;
      if (x < 0 || x >= V) {
        uflags |= SPEC_FLAG_BAD_TOKEN;
      } else {
        const float zpx = gather_z<TE>(sp, x, P.slice, cluster);
        const float zqx = dq.onehot ? 0.f : gather_z<TE>(sq, x, P.slice, cluster);
        const float qx = prob(dq, zqx, x);
        if (!(qx > 0.f)) {
          uflags |= SPEC_FLAG_ZERO_Q;
        } else {
          const float px = residual ? weight(dp, dq, 1, c, zpx, zqx, x) / Wcur : prob(dp, zpx, x);
          const float alpha = fminf(1.f, px / qx);
          acc = u < alpha;
        }
      }
      if (acc) {
        next = child;
        break;
      }
      const float cn = residual ? c + Wcur : 1.f;
      const float W = cluster_total<TE>(dp, dq, 1, cn, sp, sq, v0, len, ctl, cluster, C, xround);
      if (W > 0.f) {
        residual = 1;
        c = cn;
        Wcur = W;
        have_parts = true;
      } else {
        uflags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
        have_parts = false;  // ctl.parts now holds the rejected candidate's totals
      }
    }
    if (next < 0) {
      // ---- inverse-CDF draw over the cluster
      float Z;
      if (have_parts) {
        Z = Wcur;
      } else {
        Z = cluster_total<TE>(dp, dq, residual, residual ? c : 0.f, sp, sq, v0, len, ctl,
                              cluster, C, xround);
      }
      const float u = unit_uniform(P, seq, node, 1);
      const float t = u * Z;
      int owner = -1;
      float acc = 0.f, trel = INFINITY;
      for (int r = 0; r < C; ++r) {
        const float pr = ctl.parts[r];
        if (acc + pr > t) {
          owner = r;
          trel = t - acc;
          break;
        }
        acc += pr;
      }
      if (owner < 0) {
        for (int r = C - 1; r >= 0; --r)
          if (ctl.parts[r] > 0.f) {
            owner = r;
            break;
          }
        trel = INFINITY;
      }
      if (rank == owner) {
        const int tok = cta_search<TE>(dp, dq, residual, c, sp, sq, v0, len, trel, ctl);
        if (tid == 0) cluster.map_shared_rank(&ctl.token, 0)[0] = tok;
      }
      kind = has_children ? 2 : 0;
      total = Z;
    }
  }
  cluster.sync();

  // ---- publish this unit's outcome; the last unit of the sequence stitches
  if (rank == 0) {
    if (tid == 0) {
      if (next < 0 && !dp.onehot) token = ctl.token;
      UnitOut o;
      o.next = next;
      o.token = token;
      o.flags = uflags;
      o.pad = 0;
      P.outs[unit] = o;
      UnitStats st;
      st.p = dp;
      st.q = dq;
      st.c = residual ? c : 0.f;
      st.total = total;
      st.kind = kind;
      st.node = node;
      P.stats[unit] = st;
      __threadfence();
      const unsigned prev = atomicAdd(P.counters + seq, 1u);
      ctl.is_last = prev == static_cast<unsigned>(P.ups - 1);
    }
    __syncthreads();
    if (ctl.is_last) {
      __threadfence();
      const long long ubase = static_cast<long long>(seq) * P.ups;
      if (P.mode == kModeChain) {
        if (tid < 32) {
          const int lane = tid;
          int j = -1;
          for (int base = 0; base <= P.gamma && j < 0; base += 32) {
            const int i = base + lane;
            const bool stop = i <= P.gamma && __ldcg(&P.outs[ubase + i].next) < 0;
            const unsigned b = __ballot_sync(0xFFFFFFFFu, stop);
            if (b) j = base + __ffs(b) - 1;
          }
          uint32_t f = 0u;
          for (int i = lane; i <= j; i += 32) f |= __ldcg(&P.outs[ubase + i].flags);
          f = warp_or(f);
          const int jtok = __ldcg(&P.outs[ubase + j].token);
          const long long obase = static_cast<long long>(seq) * (P.gamma + 1);
          for (int i = lane; i <= P.gamma; i += 32) {
            int v = -1;
            if (i < j) v = __ldg(P.tokens + static_cast<long long>(seq) * P.gamma + i);
            else if (i == j) v = jtok;
            P.out_tokens[obase + i] = v;
          }
          if (lane == 0) {
            P.out_num[seq] = j;
            if (P.out_flags) P.out_flags[seq] = f;
            P.final_unit[seq] = static_cast<int>(ubase + j);
            P.counters[seq] = 0u;
          }
        }
      } else {
        // validate the tree: links, then depth by pointer jumping
        const int N = P.ups;
        const int32_t *par = P.parent + ubase;
        int *anc = reinterpret_cast<int *>(smem_raw + P.ctl_bytes);
        int *dep = anc + N;
        uint32_t bad = 0u;
        for (int n = tid; n < N; n += kThreads) {
          const int a = __ldg(par + n);
          if (n == 0 ? a != -1 : !(a >= 0 && a < n)) bad = 1u;
          anc[n] = n == 0 ? 0 : a;
          dep[n] = n == 0 ? 0 : 1;
        }
        bad = warp_or(bad);
        if ((tid & 31) == 0) ctl.red_u[tid >> 5] = bad;
        __syncthreads();
        bad = 0u;
        for (int w = 0; w < kWarps; ++w) bad |= ctl.red_u[w];
        __syncthreads();
        uint32_t tflags = bad ? SPEC_FLAG_BAD_TREE : 0u;
        if (!bad) {
          for (int span = 1; span < N; span <<= 1) {
            int la[16], ld[16];
            int cnt = 0;
            for (int n = tid; n < N && cnt < 16; n += kThreads, ++cnt) {
              const int a = anc[n];
              la[cnt] = anc[a];
              ld[cnt] = dep[n] + dep[a];
            }
            __syncthreads();
            cnt = 0;
            for (int n = tid; n < N && cnt < 16; n += kThreads, ++cnt) {
              anc[n] = la[cnt];
              dep[n] = ld[cnt];
            }
            __syncthreads();
          }
          uint32_t deep = 0u;
          for (int n = tid; n < N; n += kThreads)
            if (dep[n] > P.max_depth) deep = 1u;
          deep = warp_or(deep);
          if ((tid & 31) == 0) ctl.red_u[tid >> 5] = deep;
          __syncthreads();
          deep = 0u;
          for (int w = 0; w < kWarps; ++w) deep |= ctl.red_u[w];
          __syncthreads();
          if (deep) tflags = SPEC_FLAG_DEPTH;
        }
        const int width = P.max_depth + 1;
        const long long obase = static_cast<long long>(seq) * width;
        if (tflags) {
          for (int i = tid; i < width; i += kThreads) {
            P.out_path[obase + i] = -1;
            P.out_tokens[obase + i] = -1;
          }
          if (tid == 0) {
            P.out_num[seq] = -1;
            if (P.out_flags) P.out_flags[seq] = tflags;
            P.final_unit[seq] = -1;
          }
        } else if (tid == 0) {
          int cur = 0, k = 0;
          uint32_t f = __ldcg(&P.outs[ubase].flags);
          P.out_path[obase] = 0;
          int nx = __ldcg(&P.outs[ubase].next);
          while (nx > cur && nx < N && k < P.max_depth) {
            ++k;
            cur = nx;
            P.out_path[obase + k] = cur;
            P.out_tokens[obase + k - 1] = __ldg(P.tokens + ubase + cur);
            f |= __ldcg(&P.outs[ubase + cur].flags);
            nx = __ldcg(&P.outs[ubase + cur].next);
          }
          P.out_tokens[obase + k] = __ldcg(&P.outs[ubase + cur].token);
          for (int i = k + 1; i < width; ++i) {
            P.out_path[obase + i] = -1;
            P.out_tokens[obase + i] = -1;
          }
          P.out_num[seq] = k;
          if (P.out_flags) P.out_flags[seq] = f;
          P.final_unit[seq] = static_cast<int>(ubase + cur);
        }
        if (tid == 0) P.counters[seq] = 0u;
      }
    }
  }
}

// ---------------------------------------------------------------------------
// residual output: the distribution each sequence's final token came from
// ---------------------------------------------------------------------------

template <typename TE>
__global__ void __launch_bounds__(kThreads) residual_kernel(const Params P, float *out) {
  const int seq = blockIdx.y;
  const int V = P.V;
  const int u = P.final_unit[seq];
  float *o = out + static_cast<long long>(seq) * V;
  const int vbeg = blockIdx.x * kThreads * 8;
  if (u < 0) {
    for (int v = vbeg + threadIdx.x; v < min(V, vbeg + kThreads * 8); v += kThreads) o[v] = 0.f;
    return;
  }
  const UnitStats st = P.stats[u];
  const int node = st.node;
  const int s2 = u / P.ups;
  long long prow, qrow;
  if (P.mode == kModeChain) {
    prow = static_cast<long long>(s2) * (P.gamma + 1) + node;
    qrow = static_cast<long long>(s2) * P.gamma + node;
  } else {
    prow = static_cast<long long>(s2) * P.ups + node;
    qrow = prow;
  }
  const TE *gp = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE)));
  const TE *gq = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE)));
  const int residual = st.c > 0.f;
  for (int v = vbeg + threadIdx.x; v < min(V, vbeg + kThreads * 8); v += kThreads) {
    float r = 0.f;
    if (st.kind == 1) {
      r = v == st.p.a ? 1.f : 0.f;
    } else if (st.kind == 2) {
      const float zp = st.p.onehot ? 0.f : to_f32(gp[v]);
      const float zq = (residual && !st.q.onehot) ? to_f32(gq[v]) : 0.f;
      r = weight(st.p, st.q, residual, st.c, zp, zq, v) / st.total;
    }
    o[v] = r;
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename TE, bool kVec>
cudaError_t launch_units_t(const Params &P, int n_units, size_t smem, cudaStream_t stream) {
  auto kern = unit_kernel<TE, kVec>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  if (P.cluster > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(n_units) * P.cluster, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = P.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

cudaError_t launch_units(const Params &P, int esize, bool vec, int n_units, size_t smem,
                         cudaStream_t stream) {
  if (esize == 2)
    return vec ? launch_units_t<uint16_t, true>(P, n_units, smem, stream)
               : launch_units_t<uint16_t, false>(P, n_units, smem, stream);
  return vec ? launch_units_t<float, true>(P, n_units, smem, stream)
             : launch_units_t<float, false>(P, n_units, smem, stream);
}

cudaError_t launch_residual(const Params &P, int esize, float *out, cudaStream_t stream) {
  dim3 grid((P.V + kThreads * 8 - 1) / (kThreads * 8), P.nseq, 1);
  if (esize == 2)
    residual_kernel<uint16_t><<<grid, kThreads, 0, stream>>>(P, out);
  else
    residual_kernel<float><<<grid, kThreads, 0, stream>>>(P, out);
  return cudaGetLastError();
}

}  // namespace sv
