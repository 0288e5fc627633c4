// Per-position overlap of a draft chain: beta_i = sum_v min(p_i(v), q_i(v)).
//
// whoami-wesleyyou.top "Speculative Decoding" notes, section "Correction 为什么
// 用正残差": beta := sum_x min(p(x), q(x)) is the acceptance rate of one
// position (Z = 1 - beta is the mass of the residual [p - q]_+); beta = 1
// when p = q.
//
// A cluster of C CTAs per (sequence, position), C in {1, 2, 4}; CTA r owns
// the slice [r S, (r + 1) S) of the vocabulary, S a multiple of 8.  C is the
// smallest size whose slices of the row pair take at most 64 KB (4 when none
// does), raised while the grid would hold fewer than three CTAs per SM.  The
// slices of the CTAs in flight (at most about 80 MB) stay in the L2 between
// the two passes, so the pair leaves HBM once.  (Clusters of 8 measured slower:
// the per-CTA merges and barriers then outweigh the work.)
//
// Pass 1, per row with temperature T > 0: each thread loads four groups of 8
// at a time, takes their max (packed bf16x2 max), rescales its running sum
// when the max grew, and adds 2^(z k - m k) with k = log2(e) / T (packed
// fp32x2 fma, special-function exp2).  The (m k, S) pairs are merged over the
// block and then over the cluster through distributed shared memory, in rank
// order, so every CTA holds the same row statistics.  A greedy row (T = 0, or
// a temperature that is not finite or negative) instead takes its finite
// argmax, lowest index among equals; so does a row whose statistics show a
// NaN or an infinite logit, in a second round.  Such rows are the one-hot
// distribution at that argmax.
//
// Pass 2 sums min(p, q) over the slice in the log domain, one exponential per
// column: min(p, q) = 2^min(lp, lq) with l = z k - (m k + log2 S).  Partial
// sums run in fp32 over a few terms each, then in double-float and double.
// When a side is one-hot no second pass is needed: beta is the other side's
// probability at that index.
#include <climits>

#include "common.cuh"
#include "ops.cuh"
#include "precise.cuh"
#include "slice_rows.cuh"

namespace sv {

namespace {

constexpr int kOvCluster = 4;
constexpr size_t kSliceTarget = 64 * 1024;  // both rows' slices, per CTA

// Statistics of one row: for T > 0, mk = (max finite-or-inf logit) * k and
// S = sum 2^(z k - mk) (NaN when a NaN was summed); for the argmax, the finite
// maximum av, its lowest index ai (INT_MAX: none) and bad (a NaN or +inf).
struct RowStat {
  float mk;
  Df S;
  float av;
  int ai;
  int bad;
};

__device__ __forceinline__ RowStat empty_stat() {
  return RowStat{-INFINITY, Df{0.f, 0.f}, -INFINITY, INT_MAX, 0};
}

// One thread's (mk, S) over the groups t, t + kThreads, ... of a slice of n
// entries, kBatch groups per step: the batch's max, a rescale of the running
// sum when it grew, then the batch's exponentials in four independent pair
// chains (each at most 4 * kBatch * 4 terms before it is folded into S).
constexpr int kBatch = 4;

template <typename TE>
__device__ RowStat thread_sum(const TE *g, int n, float k, bool vec) {
  const int ngroups = (n + 7) / 8;
  const uint64_t k2 = pack2(k, k);
  float m = -INFINITY, mk = -INFINITY;
  Df S{0.f, 0.f};
  bool nan = false;
  for (int j0 = threadIdx.x; j0 < ngroups; j0 += kThreads * kBatch) {
    Group<TE> x[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      const int j = j0 + b * kThreads;
      x[b] = load_group<TE>(g, 8 * j, n, vec && 8 * j + 8 <= n);
    }
    float bm = group_max(x[0]);
#pragma unroll
    for (int b = 1; b < kBatch; ++b) bm = fmaxf(bm, group_max(x[b]));
    if (bm == -INFINITY) {  // only -inf and NaN (the max skips NaN)
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
#pragma unroll
        for (int e = 0; e < 8; ++e) nan |= entry(x[b], e) != entry(x[b], e);
      continue;
    }
    if (bm > m) {
      const float nmk = bm * k;
      if (m > -INFINITY) S = df_mul(S, Df{fast_exp2(mk - nmk), 0.f});
      m = bm;
      mk = nmk;
    }
    const uint64_t nm2 = pack2(-mk, -mk);
    uint64_t a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
#pragma unroll
      for (int i = 0; i < 4; ++i)
        a[i] = fadd2(a[i], ex2_pair(ffma2(pair_of(x[b], 2 * i), k2, nm2)));
    S = df_add(S, Df{hsum2(fadd2(fadd2(a[0], a[1]), fadd2(a[2], a[3]))), 0.f});
  }
  RowStat r = empty_stat();
  r.mk = mk;
  r.S = S;
  if (nan) r.S.hi = __int_as_float(0x7FC00000);
  return r;
}

// One thread's finite argmax and non-finite flag (slice_argmax) as a RowStat.
template <typename TE>
__device__ RowStat thread_argmax(const TE *g, int n, int lo, bool vec) {
  const ArgStat a = slice_argmax<TE>(g, n, lo, vec);
  RowStat r = empty_stat();
  r.av = a.av;
  r.ai = a.ai;
  r.bad = a.bad;
  return r;
}

// a += b.  (mk, S) pairs merge as S_a 2^(mk_a - M) + S_b 2^(mk_b - M); a NaN
// sum or an infinite max carries through as NaN or +inf.
__device__ void merge_into(RowStat &a, const RowStat &b) {
  if (b.mk > a.mk) {
    if (a.mk > -INFINITY) a.S = df_mul(a.S, Df{fast_exp2(a.mk - b.mk), 0.f});
    a.S = df_add(a.S, b.S);
    a.mk = b.mk;
  } else if (b.mk > -INFINITY) {
    a.S = df_add(a.S, df_mul(b.S, Df{fast_exp2(b.mk - a.mk), 0.f}));
  } else if (b.S.hi != b.S.hi) {
    a.S = b.S;
  }
  argmax_merge(a.av, a.ai, b.av, b.ai);
  a.bad |= b.bad;
}

// Distribution of a row: one-hot at `a`, or p(z) = 2^(z k - C) with the
// constant C = mk + log2 S split into C + C_lo.
struct Side {
  int onehot, a, flagged;
  float k, C, C_lo;
  __device__ __forceinline__ float log2p(float z) const { return fmaf(z, k, -C) - C_lo; }
  __device__ float prob(float z, int v) const {
    if (onehot) return v == a ? 1.f : 0.f;
    return z > -INFINITY ? fast_exp2(log2p(z)) : 0.f;
  }
};

// Whether a T > 0 row's merged statistics are usable (finite max, a positive
// finite sum: no NaN or infinite logit, at least one finite one).
__device__ __forceinline__ bool stats_ok(const RowStat &st) {
  const double S = df_to_double(st.S);
  return st.mk > -INFINITY && st.mk < INFINITY && S > 0.0 && S < INFINITY;
}

__device__ Side make_side(const RowStat &st, float T, bool sampled) {
  Side d;
  const bool tbad = !(T >= 0.f) || T == INFINITY;
  d.a = st.ai == INT_MAX ? 0 : st.ai;
  d.k = 0.f;
  d.C = d.C_lo = 0.f;
  if (sampled && stats_ok(st)) {
    d.onehot = 0;
    d.flagged = 0;
    d.k = kLog2e / T;
    const double C = static_cast<double>(st.mk) + log2(df_to_double(st.S));
    d.C = static_cast<float>(C);
    d.C_lo = static_cast<float>(C - static_cast<double>(d.C));
  } else {
    d.onehot = 1;
    d.flagged = tbad || st.bad || st.ai == INT_MAX;
  }
  return d;
}

struct OverlapSmem {
  RowStat warp[2][kWarps];
  RowStat slice[2][kOvCluster][2];  // [round][rank][row], written by that rank
  Df part[kWarps];
  double bpart[kOvCluster];  // every rank's partial beta (read by rank 0)
  RowStat row[2];            // merged statistics
  int redo[2];               // a sampled row whose statistics are unusable
  Side side[2];              // the two rows' distributions
};

// Merges the threads' statistics of both rows over the block, stores each
// rank's result into every rank's shared memory (slot `round`), waits on the
// cluster barrier and merges the C slices in rank order into sm.row.  The
// first round's wait also covers the arrival made at the kernel's start, so
// no CTA's shared memory is written before that CTA runs.
__device__ void cluster_merge(RowStat r[2], OverlapSmem &sm, cg::cluster_group &cluster, int rank,
                              int C, int round) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int x = 0; x < 2; ++x) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      RowStat o;
      o.mk = __shfl_xor_sync(0xFFFFFFFFu, r[x].mk, off);
      o.S.hi = __shfl_xor_sync(0xFFFFFFFFu, r[x].S.hi, off);
      o.S.lo = __shfl_xor_sync(0xFFFFFFFFu, r[x].S.lo, off);
      o.av = __shfl_xor_sync(0xFFFFFFFFu, r[x].av, off);
      o.ai = __shfl_xor_sync(0xFFFFFFFFu, r[x].ai, off);
      o.bad = __shfl_xor_sync(0xFFFFFFFFu, r[x].bad, off);
      merge_into(r[x], o);
    }
    if (lane == 0) sm.warp[x][warp] = r[x];
  }
  __syncthreads();
  if (round == 0) cluster_wait();
  if (threadIdx.x < 2) {
    const int x = threadIdx.x;
    RowStat a = empty_stat();
    for (int w = 0; w < kWarps; ++w) merge_into(a, sm.warp[x][w]);
    for (int d = 0; d < C; ++d) cluster.map_shared_rank(&sm.slice[round][rank][x], d)[0] = a;
  }
  cluster_sync_all();
  if (threadIdx.x < 2) {
    const int x = threadIdx.x;
    RowStat a = empty_stat();
    for (int d = 0; d < C; ++d) merge_into(a, sm.slice[round][d][x]);
    sm.row[x] = a;
  }
  __syncthreads();
}

template <typename TE>
__global__ void __launch_bounds__(kThreads) overlap_kernel(
    const TE *target, long long ld_t, const TE *draft, long long ld_d, int gamma, int V, int S_e,
    const float *Tp, const float *Tq, float *out_beta, uint32_t *out_flags) {
  __shared__ OverlapSmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  cluster_arrive_relaxed();  // waited on before the first remote store
  const int unit = blockIdx.x / C;
  const int seq = unit / gamma, pos = unit - seq * gamma;
  const TE *gp = target + (static_cast<long long>(seq) * (gamma + 1) + pos) * ld_t;
  const TE *gq = draft + (static_cast<long long>(seq) * gamma + pos) * ld_d;
  const bool vec = ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(gq)) & 15u) == 0;
  const int lo = rank * S_e;
  const int n = max(0, min(V - lo, S_e));
  const TE *sp = gp + lo, *sq = gq + lo;
  const float T[2] = {__ldg(Tp + seq), __ldg(Tq + seq)};
  bool sampled[2];
#pragma unroll
  for (int x = 0; x < 2; ++x) sampled[x] = T[x] > 0.f && T[x] != INFINITY;
  // pass 1: (mk, S) of a sampled row, the argmax of a greedy one
  RowStat r[2];
  r[0] = sampled[0] ? thread_sum<TE>(sp, n, kLog2e / T[0], vec)
                    : thread_argmax<TE>(sp, n, lo, vec);
  r[1] = sampled[1] ? thread_sum<TE>(sq, n, kLog2e / T[1], vec)
                    : thread_argmax<TE>(sq, n, lo, vec);
  cluster_merge(r, sm, cluster, rank, C, 0);
  // A sampled row whose statistics are unusable becomes the one-hot at its
  // finite argmax: a second round, uniform over the cluster (every CTA holds
  // the same merged statistics).  Double-precision work stays on two threads.
  if (threadIdx.x < 2) {
    const int x = threadIdx.x;
    sm.redo[x] = sampled[x] && !stats_ok(sm.row[x]);
    if (!sm.redo[x]) sm.side[x] = make_side(sm.row[x], T[x], sampled[x]);
  }
  __syncthreads();
  const bool redo[2] = {sm.redo[0] != 0, sm.redo[1] != 0};
  if (redo[0] || redo[1]) {
    r[0] = redo[0] ? thread_argmax<TE>(sp, n, lo, vec) : empty_stat();
    r[1] = redo[1] ? thread_argmax<TE>(sq, n, lo, vec) : empty_stat();
    cluster_merge(r, sm, cluster, rank, C, 1);
    if (threadIdx.x < 2 && redo[threadIdx.x])
      sm.side[threadIdx.x] = make_side(sm.row[threadIdx.x], T[threadIdx.x], false);
    __syncthreads();
  }
  const Side dp = sm.side[0], dq = sm.side[1];
  const bool flagged = dp.flagged || dq.flagged;
  if (dp.onehot || dq.onehot) {
    if (rank == 0 && threadIdx.x == 0) {
      // one side is one index: beta is the other side's probability there
      double beta;
      if (dp.onehot && dq.onehot) beta = dp.a == dq.a ? 1.0 : 0.0;
      else if (dp.onehot) beta = dq.prob(to_f32(gq[dp.a]), dp.a);
      else beta = dp.prob(to_f32(gp[dq.a]), dq.a);
      out_beta[unit] = static_cast<float>(beta);
      if (out_flags && flagged) atomicOr(out_flags + seq, SPEC_FLAG_NONFINITE);
    }
    return;
  }
  // pass 2: sum over the slice of min(p, q) = 2^min(lp, lq)
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t kp2 = pack2(dp.k, dp.k), kq2 = pack2(dq.k, dq.k);
  const uint64_t cp2 = pack2(-dp.C, -dp.C), cq2 = pack2(-dq.C, -dq.C);
  const uint64_t clp2 = pack2(-dp.C_lo, -dp.C_lo), clq2 = pack2(-dq.C_lo, -dq.C_lo);
  Df acc{0.f, 0.f};
  const int ngroups = (n + 7) / 8;
  constexpr int kB2 = kBatch / 2;  // both rows' groups in registers
  for (int j0 = threadIdx.x; j0 < ngroups; j0 += kThreads * kB2) {
    Group<TE> xp[kB2], xq[kB2];
#pragma unroll
    for (int b = 0; b < kB2; ++b) {
      const int j = j0 + b * kThreads;
      const bool fast = vec && 8 * j + 8 <= n;
      xp[b] = load_group<TE>(sp, 8 * j, n, fast);
      xq[b] = load_group<TE>(sq, 8 * j, n, fast);
    }
    uint64_t a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int b = 0; b < kB2; ++b)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float lp0, lp1, lq0, lq1;
        unpack2(fadd2(ffma2(pair_of(xp[b], 2 * i), kp2, cp2), clp2), lp0, lp1);
        unpack2(fadd2(ffma2(pair_of(xq[b], 2 * i), kq2, cq2), clq2), lq0, lq1);
        a[i] = fadd2(a[i], pack2(fast_exp2(fminf(lp0, lq0)), fast_exp2(fminf(lp1, lq1))));
      }
    acc = df_add(acc, Df{hsum2(fadd2(fadd2(a[0], a[1]), fadd2(a[2], a[3]))), 0.f});
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    acc = df_add(acc, Df{__shfl_xor_sync(0xFFFFFFFFu, acc.hi, off),
                         __shfl_xor_sync(0xFFFFFFFFu, acc.lo, off)});
  if (lane == 0) sm.part[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    double b = 0.0;
    for (int w = 0; w < kWarps; ++w) b += df_to_double(sm.part[w]);
    cluster.map_shared_rank(&sm.bpart[rank], 0)[0] = b;
  }
  cluster_sync_all();
  if (rank == 0 && threadIdx.x == 0) {
    double beta = 0.0;
    for (int d = 0; d < C; ++d) beta += sm.bpart[d];
    out_beta[unit] = static_cast<float>(beta);
    if (out_flags && flagged) atomicOr(out_flags + seq, SPEC_FLAG_NONFINITE);
  }
}

template <typename TE>
cudaError_t launch_typed(const void *target, long long ld_t, const void *draft, long long ld_d,
                         int gamma, int V, long long units, const float *Tp, const float *Tq,
                         float *out_beta, uint32_t *out_flags, cudaStream_t stream) {
  auto slice = [V](int c) { return ((V + c - 1) / c + 7) / 8 * 8; };
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int C = 1;
  while (C < kOvCluster && 2ull * slice(C) * sizeof(TE) > kSliceTarget) C *= 2;
  while (C < kOvCluster && units * C < 3ll * sms) C *= 2;
  const int S_e = slice(C);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, overlap_kernel<TE>, static_cast<const TE *>(target), ld_t,
                            static_cast<const TE *>(draft), ld_d, gamma, V, S_e, Tp, Tq, out_beta,
                            out_flags);
}

}  // namespace

cudaError_t launch_overlap(const void *target, long long ld_t, const void *draft, long long ld_d,
                           int esize, int B, int gamma, int V, const float *Tp, const float *Tq,
                           float *out_beta, uint32_t *out_flags, cudaStream_t stream) {
  const long long units = static_cast<long long>(B) * gamma;
  if (units == 0) return cudaSuccess;
  if (units * kOvCluster > 0x7FFFFFFFll) return cudaErrorInvalidValue;
  if (esize == 2)
    return launch_typed<uint16_t>(target, ld_t, draft, ld_d, gamma, V, units, Tp, Tq, out_beta,
                                  out_flags, stream);
  return launch_typed<float>(target, ld_t, draft, ld_d, gamma, V, units, Tp, Tq, out_beta,
                             out_flags, stream);
}

}  // namespace sv
