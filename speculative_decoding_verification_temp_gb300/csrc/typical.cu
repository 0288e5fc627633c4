// Typical acceptance of a draft chain: an approximate acceptance rule whose
// output law is not the target's.
//
// whoami-wesleyyou.top "Speculative Decoding" notes, section "Medusa-1 与
// typical acceptance": draft token x_i passes when p_i(x_i) > min(epsilon,
// delta exp(-H(p_i))), H the entropy of the target's distribution at that
// position; the longest passing prefix is kept and the token after it is the
// target's greedy choice, accepted without a test.  jennyma11.github.io "11.3
// Self-Draft: Medusa、EAGLE-2/3 与 Draft Tree", section 11.3.1: an approximate
// acceptance mode, not the exact one.
//
// Each test needs only its own target row, so the rows are independent:
//
// typical_row_kernel: a cluster of C CTAs per target row (B (gamma + 1) rows),
// CTA r owning the vocabulary slice [r S, (r + 1) S).  Each thread loads four
// groups of 8 at a time and keeps, relative to its running max m,
// S1 = sum 2^t and S2 = sum 2^t t with t = z k - m k, k = log2(e) / T
// (packed bf16x2 max, packed fp32x2 fma, special-function exp2), and the
// lowest index of its max.  The statistics merge over the block and then the
// cluster (distributed shared memory, rank order).  Then
//   H = ln 2 (log2 S1 - S2 / S1),   p(x) = 2^(z_x k - m k - log2 S1),
// in double on one thread, and the row's result (pass bit, flags, greedy
// token) goes to the workspace.  A greedy row (T = 0, or a temperature that
// is not finite or negative) is the one-hot at its finite argmax (H = 0); so
// is a row whose statistics show a NaN or infinite logit (flagged), found in a
// second, argmax-only round.
//
// typical_decide_kernel: one thread per sequence walks its rows: the first
// row that fails (or the bonus row) gives the greedy token and ends the chain.
#include <climits>

#include "common.cuh"
#include "ops.cuh"
#include "precise.cuh"
#include "slice_rows.cuh"

namespace sv {

size_t chain_rows_ctl_bytes();
cudaError_t launch_typical_rows(const Params &P, int esize, size_t smem, cudaStream_t stream);

namespace {

constexpr int kTyCluster = 4;
constexpr size_t kSliceTarget = 64 * 1024;  // one row's slice, per CTA
constexpr int kBatch = 4;
constexpr int kPass = 1;  // row result bit: the draft token passed its test

// Row statistics: mk = m k, S1 = sum 2^t, S2 = sum 2^t t (t = z k - mk) for a
// sampled row; av, ai = the max and its lowest index; bad = a NaN or +inf.
struct TyStat {
  float mk;
  Df S1, S2;
  float av;
  int ai;
  int bad;
};

__device__ __forceinline__ TyStat ty_empty() {
  return TyStat{-INFINITY, Df{0.f, 0.f}, Df{0.f, 0.f}, -INFINITY, INT_MAX, 0};
}

__device__ __forceinline__ Df df_scale(Df a, float f) { return df_mul(a, Df{f, 0.f}); }

// (S1, S2) re-expressed relative to a max that grew by -d (d = mk_old - mk_new
// <= 0): S1' = f S1, S2' = f (S2 + d S1), f = 2^d.
__device__ __forceinline__ void ty_rescale(Df &S1, Df &S2, float d) {
  const float f = fast_exp2(d);
  S2 = df_scale(df_add(S2, df_scale(S1, d)), f);
  S1 = df_scale(S1, f);
}

// max(t, -150) that keeps a NaN: 2^-150 flushes to zero, so a -inf logit
// adds 0 to S1 and 0 (not 0 * -inf) to S2.
__device__ __forceinline__ float clamp_t(float t) { return t < -150.f ? -150.f : t; }

// One thread's statistics of a sampled row's slice of n entries starting at
// vocabulary index lo.
template <typename TE>
__device__ TyStat thread_stats(const TE *g, int n, int lo, float k, bool vec) {
  const int ngroups = (n + 7) / 8;
  const uint64_t k2 = pack2(k, k);
  TyStat r = ty_empty();
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
    if (bm > r.av) {
      // the lowest index of the new max: earlier batches and groups hold
      // lower indices, so the first match in (b, e) order
      int ai = INT_MAX;
#pragma unroll
      for (int b = kBatch - 1; b >= 0; --b)
#pragma unroll
        for (int e = 7; e >= 0; --e)
          if (entry(x[b], e) == bm) ai = lo + 8 * (j0 + b * kThreads) + e;
      const float nmk = bm * k;
      if (r.av > -INFINITY) ty_rescale(r.S1, r.S2, r.mk - nmk);
      r.av = bm;
      r.ai = ai;
      r.mk = nmk;
    }
    const uint64_t nm2 = pack2(-r.mk, -r.mk);
    uint64_t a1[4] = {0ull, 0ull, 0ull, 0ull}, a2[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
    for (int b = 0; b < kBatch; ++b)
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        float t0, t1;
        unpack2(ffma2(pair_of(x[b], 2 * i), k2, nm2), t0, t1);
        const uint64_t t2 = pack2(clamp_t(t0), clamp_t(t1));
        const uint64_t w2 = ex2_pair(t2);
        a1[i] = fadd2(a1[i], w2);
        a2[i] = ffma2(w2, t2, a2[i]);
      }
    r.S1 = df_add(r.S1, Df{hsum2(fadd2(fadd2(a1[0], a1[1]), fadd2(a1[2], a1[3]))), 0.f});
    r.S2 = df_add(r.S2, Df{hsum2(fadd2(fadd2(a2[0], a2[1]), fadd2(a2[2], a2[3]))), 0.f});
  }
  if (nan) r.S1.hi = __int_as_float(0x7FC00000);
  return r;
}

template <typename TE>
__device__ TyStat thread_argmax(const TE *g, int n, int lo, bool vec) {
  const ArgStat a = slice_argmax<TE>(g, n, lo, vec);
  TyStat r = ty_empty();
  r.av = a.av;
  r.ai = a.ai;
  r.bad = a.bad;
  return r;
}

// a += b.  A NaN sum or an infinite max carries through.
__device__ void ty_merge(TyStat &a, const TyStat &b) {
  if (b.mk > a.mk) {
    if (a.mk > -INFINITY) ty_rescale(a.S1, a.S2, a.mk - b.mk);
    a.S1 = df_add(a.S1, b.S1);
    a.S2 = df_add(a.S2, b.S2);
    a.mk = b.mk;
  } else if (b.mk > -INFINITY) {
    Df S1 = b.S1, S2 = b.S2;
    ty_rescale(S1, S2, b.mk - a.mk);
    a.S1 = df_add(a.S1, S1);
    a.S2 = df_add(a.S2, S2);
  } else if (b.S1.hi != b.S1.hi) {
    a.S1 = b.S1;
  }
  argmax_merge(a.av, a.ai, b.av, b.ai);
  a.bad |= b.bad;
}

__device__ __forceinline__ bool ty_ok(const TyStat &st) {
  const double S1 = df_to_double(st.S1);
  return st.mk > -INFINITY && st.mk < INFINITY && S1 > 0.0 && S1 < INFINITY;
}

struct TySmem {
  TyStat warp[kWarps];
  TyStat slice[2][kTyCluster];  // [round][rank], written by that rank
  TyStat row;
  int redo;
};

// Block merge, every rank's result into every rank's shared memory (slot
// `round`), a cluster barrier, and the merge in rank order into sm.row.  The
// first round's wait pairs with the arrival made at the kernel's start.
__device__ void ty_cluster_merge(TyStat r, TySmem &sm, cg::cluster_group &cluster, int rank,
                                 int C, int round) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    TyStat o;
    o.mk = __shfl_xor_sync(0xFFFFFFFFu, r.mk, off);
    o.S1.hi = __shfl_xor_sync(0xFFFFFFFFu, r.S1.hi, off);
    o.S1.lo = __shfl_xor_sync(0xFFFFFFFFu, r.S1.lo, off);
    o.S2.hi = __shfl_xor_sync(0xFFFFFFFFu, r.S2.hi, off);
    o.S2.lo = __shfl_xor_sync(0xFFFFFFFFu, r.S2.lo, off);
    o.av = __shfl_xor_sync(0xFFFFFFFFu, r.av, off);
    o.ai = __shfl_xor_sync(0xFFFFFFFFu, r.ai, off);
    o.bad = __shfl_xor_sync(0xFFFFFFFFu, r.bad, off);
    ty_merge(r, o);
  }
  if (lane == 0) sm.warp[warp] = r;
  __syncthreads();
  if (round == 0) cluster_wait();
  if (threadIdx.x == 0) {
    TyStat a = ty_empty();
    for (int w = 0; w < kWarps; ++w) ty_merge(a, sm.warp[w]);
    for (int d = 0; d < C; ++d) cluster.map_shared_rank(&sm.slice[round][rank], d)[0] = a;
  }
  cluster_sync_all();
  if (threadIdx.x == 0) {
    TyStat a = ty_empty();
    for (int d = 0; d < C; ++d) ty_merge(a, sm.slice[round][d]);
    sm.row = a;
  }
  __syncthreads();
}

template <typename TE>
__global__ void __launch_bounds__(kThreads) typical_row_kernel(
    const TE *target, long long ld_t, int gamma, int V, int S_e, const float *Tp,
    const int32_t *tokens, float epsilon, float delta, int2 *rows_out) {
  __shared__ TySmem sm;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = static_cast<int>(cluster.block_rank());
  const int C = static_cast<int>(cluster.num_blocks());
  cluster_arrive_relaxed();  // waited on before the first remote store
  const int row = blockIdx.x / C;  // seq * (gamma + 1) + i
  const int seq = row / (gamma + 1), i = row - seq * (gamma + 1);
  const TE *g = target + static_cast<long long>(row) * ld_t;
  const bool vec = (reinterpret_cast<uintptr_t>(g) & 15u) == 0;
  const int lo = rank * S_e;
  const int n = max(0, min(V - lo, S_e));
  const TE *sp = g + lo;
  const float T = __ldg(Tp + seq);
  const bool sampled = T > 0.f && T != INFINITY;
  const float k = sampled ? kLog2e / T : 0.f;
  ty_cluster_merge(sampled ? thread_stats<TE>(sp, n, lo, k, vec) : thread_argmax<TE>(sp, n, lo, vec),
                   sm, cluster, rank, C, 0);
  if (threadIdx.x == 0) sm.redo = sampled && !ty_ok(sm.row);
  __syncthreads();
  const bool redo = sm.redo != 0;  // the same in every CTA of the cluster
  TyStat st;
  if (redo) {
    ty_cluster_merge(thread_argmax<TE>(sp, n, lo, vec), sm, cluster, rank, C, 1);
  }
  if (rank != 0 || threadIdx.x != 0) return;
  st = sm.row;
  const bool tbad = !(T >= 0.f) || T == INFINITY;
  const bool onehot = !sampled || redo;
  const int a = st.ai == INT_MAX ? 0 : st.ai;
  uint32_t flags = 0;
  if (onehot && (tbad || st.bad || st.ai == INT_MAX)) flags |= SPEC_FLAG_NONFINITE;
  int pass = 0;
  if (i < gamma) {
    const int x = __ldg(tokens + static_cast<long long>(seq) * gamma + i);
    if (x < 0 || x >= V) {
      flags |= SPEC_FLAG_BAD_TOKEN;
    } else if (onehot) {
      const double thr = fmin(static_cast<double>(epsilon), static_cast<double>(delta));
      pass = (x == a ? 1.0 : 0.0) > thr;
    } else {
      const double S1 = df_to_double(st.S1), S2 = df_to_double(st.S2);
      const double L = log2(S1);
      const double H = 0.6931471805599453 * (L - S2 / S1);
      const double px =
          exp2(static_cast<double>(to_f32(g[x])) * static_cast<double>(k) -
               static_cast<double>(st.mk) - L);
      const double thr =
          fmin(static_cast<double>(epsilon), static_cast<double>(delta) * exp(-H));
      pass = px > thr;
    }
  }
  rows_out[row] = make_int2(static_cast<int>(flags << 8) | (pass ? kPass : 0), a);
}

__global__ void typical_decide_kernel(const int2 *rows, const int32_t *tokens, int B, int gamma,
                                      int32_t *out_num, int32_t *out_tokens, uint32_t *out_flags) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const long long base = static_cast<long long>(b) * (gamma + 1);
  uint32_t flags = 0;
  int n = gamma;
  for (int i = 0; i <= gamma; ++i) {
    const int2 r = rows[base + i];
    flags |= static_cast<uint32_t>(r.x) >> 8;
    if (i < gamma && (r.x & kPass)) {
      out_tokens[base + i] = tokens[static_cast<long long>(b) * gamma + i];
      continue;
    }
    out_tokens[base + i] = r.y;
    n = i;
    break;
  }
  for (int i = n + 1; i <= gamma; ++i) out_tokens[base + i] = -1;
  out_num[b] = n;
  if (out_flags) out_flags[b] = flags;
}

// ---------------------------------------------------------------------------
// the streaming form (16-byte aligned rows): the chain rows kernel's stream
// leaves per-warp records (max, S1, S2, lowest index of the max) of every
// target row; one warp per row merges them and runs the test
// ---------------------------------------------------------------------------

constexpr int kMWarps = 8;  // rows per CTA of the merge kernel
constexpr uint32_t kNoIdx = 0x3FFFFFFFu;
constexpr uint32_t kBadIdx = 0x80000000u;

// Lowest index of the largest finite entry of a row (one warp; 0 when none).
template <typename TE>
__device__ int warp_finite_argmax_row(const TE *g, int V) {
  const int lane = threadIdx.x & 31;
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int v = lane; v < V; v += 32) {
    const float x = to_f32(g[v]);
    if (x == x && x != INFINITY && x > bv) {
      bv = x;
      bi = v;
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
    if (v2 > bv || (v2 == bv && i2 < bi)) {
      bv = v2;
      bi = i2;
    }
  }
  return bi == INT_MAX ? 0 : bi;
}

// One warp per target row: the row's statistics from its R = cpr 8 records,
// merged in double (S1' = f S1, S2' = f (S2 + d S1) for a max that is d / k
// below the row's, f = 2^d), then the test of the row's draft token and its
// greedy token (the argmax, lowest index).
template <typename TE>
__global__ void __launch_bounds__(kMWarps * 32) typical_merge_kernel(const Params P,
                                                                     float epsilon, float delta,
                                                                     int2 *rows_out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int gamma = P.gamma, V = P.V;
  const long long nrows = static_cast<long long>(P.nseq) * (gamma + 1);
  const long long row = static_cast<long long>(blockIdx.x) * kMWarps + warp;
  if (row >= nrows) return;
  const int seq = static_cast<int>(row / (gamma + 1)), i = static_cast<int>(row % (gamma + 1));
  if (__ldcg(P.err)) {
    // a bounded wait of the rows kernel gave up: no pass, no token
    if (lane == 0) rows_out[row] = make_int2(static_cast<int>(SPEC_FLAG_TIMEOUT << 8), -1);
    return;
  }
  const float T = __ldg(P.Tp + seq);
  const bool sampled = T > 0.f && T != INFINITY;
  const float k = sampled ? kLog2e / T : 0.f;
  const int R = P.cpr * 8;
  const float4 *rec = P.trec + row * R;
  float M = -INFINITY;
  for (int x = lane; x < R; x += 32) M = fmaxf(M, __ldcg(&rec[x].x));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, off));
  double s1 = 0.0, s2 = 0.0;
  uint32_t idx = kNoIdx;
  int bad = 0;
  for (int x = lane; x < R; x += 32) {
    const float4 r = __ldcg(&rec[x]);
    const uint32_t bits = __float_as_uint(r.w);
    if (sampled) {
      if (r.y != r.y) {
        bad = 1;
      } else if (r.x > -INFINITY && M < INFINITY) {
        // the record's max is d / k below the row's (r.x - M exact for the
        // element types); single-precision scale, double sums
        const float d = __fmul_rn(__fsub_rn(r.x, M), k);
        const double f = static_cast<double>(fast_exp2(d));
        s1 += f * static_cast<double>(r.y);
        s2 += f * (static_cast<double>(r.z) + static_cast<double>(d) * static_cast<double>(r.y));
      }
    } else {
      bad |= static_cast<int>(bits >> 31);
      if (r.x == M && M > -INFINITY) idx = min(idx, (bits & ~kBadIdx) - 1u);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    s1 += __shfl_xor_sync(0xFFFFFFFFu, s1, off);
    s2 += __shfl_xor_sync(0xFFFFFFFFu, s2, off);
    idx = min(idx, __shfl_xor_sync(0xFFFFFFFFu, idx, off));
    bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
  }
  const TE *g = static_cast<const TE *>(P.target) + row * P.ld_t;
  if (sampled && M > -INFINITY && M < INFINITY) {
    // the lowest index of the max: in the first part (records run in
    // vocabulary order) whose max is the row's; its record holds it when the
    // stream computed it, else the warp searches the part
    int first = -1;
    for (int x0 = 0; x0 < R && first < 0; x0 += 32) {
      const int x = x0 + lane;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, x < R && __ldcg(&rec[x].x) == M);
      if (bal) first = x0 + __ffs(bal) - 1;
    }
    if (first >= 0) {
      const uint32_t bits = __float_as_uint(__ldcg(&rec[first].w));
      if (bits < kNoIdx) {
        idx = bits;
      } else {
        const int EW = P.chunk_elems / 8;
        const int lo = (first / 8) * P.chunk_elems + (first % 8) * EW;
        const int hi = min(V, lo + EW);
        for (int v0 = lo; v0 < hi && idx >= kNoIdx; v0 += 32 * 8) {
          uint32_t mine = kNoIdx;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int v = v0 + lane * 8 + e;
            if (v < hi && mine == kNoIdx && to_f32(g[v]) == M) mine = static_cast<uint32_t>(v);
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) mine = min(mine, __shfl_xor_sync(0xFFFFFFFFu, mine, off));
          idx = mine;
        }
      }
    }
  }
  const bool onehot = !sampled || bad || !(s1 > 0.0);
  int a;
  if (onehot && sampled && M == INFINITY) {
    a = warp_finite_argmax_row<TE>(g, V);  // +inf seen: the finite argmax
  } else {
    a = idx >= kNoIdx ? 0 : static_cast<int>(idx);
  }
  if (lane != 0) return;
  const bool tbad = !(T >= 0.f) || T == INFINITY;
  uint32_t flags = 0;
  if (onehot && (tbad || bad || (sampled && !(s1 > 0.0)) || idx >= kNoIdx))
    flags |= SPEC_FLAG_NONFINITE;
  int pass = 0;
  if (i < gamma) {
    const int x = __ldg(P.tokens + static_cast<long long>(seq) * gamma + i);
    if (x < 0 || x >= V) {
      flags |= SPEC_FLAG_BAD_TOKEN;
    } else if (onehot) {
      const double thr = fmin(static_cast<double>(epsilon), static_cast<double>(delta));
      pass = (x == a ? 1.0 : 0.0) > thr;
    } else {
      const double L = log2(s1);
      const double H = 0.6931471805599453 * (L - s2 / s1);
      const double px = exp2((static_cast<double>(to_f32(g[x])) - static_cast<double>(M)) *
                                 static_cast<double>(k) - L);
      const double thr =
          fmin(static_cast<double>(epsilon), static_cast<double>(delta) * exp(-H));
      pass = px > thr;
    }
  }
  rows_out[row] = make_int2(static_cast<int>(flags << 8) | (pass ? kPass : 0), a);
}

template <typename TE>
cudaError_t launch_rows(const void *target, long long ld_t, int B, int gamma, int V,
                        const float *Tp, const int32_t *tokens, float epsilon, float delta,
                        int2 *rows, cudaStream_t stream) {
  const long long nrows = static_cast<long long>(B) * (gamma + 1);
  auto slice = [V](int c) { return ((V + c - 1) / c + 7) / 8 * 8; };
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  int C = 1;
  while (C < kTyCluster && 1ull * slice(C) * sizeof(TE) > kSliceTarget) C *= 2;
  while (C < kTyCluster && nrows * C < 3ll * sms) C *= 2;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(nrows * C), 1, 1);
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
  return cudaLaunchKernelEx(&cfg, typical_row_kernel<TE>, static_cast<const TE *>(target), ld_t,
                            gamma, V, slice(C), Tp, tokens, epsilon, delta, rows);
}

}  // namespace

// Workspace: the error word (256 bytes), the per-row results, then the
// streaming form's records.
namespace {
constexpr size_t kTyHead = 256;
constexpr int kTyChunk = 32 * 1024;  // bytes of a chunk of the rows kernel
size_t align256(size_t x) { return (x + 255) / 256 * 256; }
}  // namespace

size_t typical_workspace_bytes(int B, int gamma, int V, int esize) {
  const size_t rows = static_cast<size_t>(B) * (gamma + 1);
  const size_t cpr = (static_cast<size_t>(V) * esize + kTyChunk - 1) / kTyChunk;
  return kTyHead + align256(rows * sizeof(int2)) + rows * cpr * 8 * sizeof(float4);
}

cudaError_t launch_typical(const void *target, long long ld_t, int esize, int B, int gamma, int V,
                           const float *Tp, const int32_t *tokens, float epsilon, float delta,
                           int32_t *out_num, int32_t *out_tokens, uint32_t *out_flags,
                           void *workspace, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  const long long nrows = static_cast<long long>(B) * (gamma + 1);
  char *ws = static_cast<char *>(workspace);
  int2 *rows = reinterpret_cast<int2 *>(ws + kTyHead);
  const bool aligned = (reinterpret_cast<uintptr_t>(target) & 15u) == 0 && (ld_t * esize) % 16 == 0;
  const int chunk = kTyChunk / esize;
  const long long cpr = (static_cast<long long>(V) + chunk - 1) / chunk;
  cudaError_t e;
  if (aligned && nrows * cpr * 8 < 0x7FFFFFFFll) {
    // the stream: every target row read once, records, then one warp per row
    e = cudaMemsetAsync(ws, 0, kTyHead, stream);
    if (e != cudaSuccess) return e;
    Params P{};
    P.nseq = B;
    P.gamma = gamma;
    P.V = V;
    P.target = target;
    P.ld_t = ld_t;
    P.Tp = Tp;
    P.tokens = tokens;
    P.err = reinterpret_cast<uint32_t *>(ws);
    P.trec = reinterpret_cast<float4 *>(ws + kTyHead + align256(nrows * sizeof(int2)));
    P.chunk_elems = chunk;
    P.cpr = static_cast<int>(cpr);
    P.ring = 2;
    P.slot_bytes = kTyChunk;
    P.first_wait = kWaitLimitCycles;
    const size_t off = (chain_rows_ctl_bytes() + 127) / 128 * 128;
    P.data_off = static_cast<int>(off);
    e = launch_typical_rows(P, esize, off + 2 * static_cast<size_t>(kTyChunk), stream);
    if (e != cudaSuccess) return e;
    const unsigned blocks = static_cast<unsigned>((nrows + kMWarps - 1) / kMWarps);
    if (esize == 2)
      typical_merge_kernel<uint16_t><<<blocks, kMWarps * 32, 0, stream>>>(P, epsilon, delta, rows);
    else
      typical_merge_kernel<float><<<blocks, kMWarps * 32, 0, stream>>>(P, epsilon, delta, rows);
    e = cudaGetLastError();
  } else {
    // unaligned rows: one cluster of CTAs per row reads its slices
    if (nrows * kTyCluster > 0x7FFFFFFFll) return cudaErrorInvalidValue;
    e = esize == 2 ? launch_rows<uint16_t>(target, ld_t, B, gamma, V, Tp, tokens, epsilon, delta,
                                           rows, stream)
                   : launch_rows<float>(target, ld_t, B, gamma, V, Tp, tokens, epsilon, delta, rows,
                                        stream);
  }
  if (e != cudaSuccess) return e;
  typical_decide_kernel<<<(B + kThreads - 1) / kThreads, kThreads, 0, stream>>>(
      rows, tokens, B, gamma, out_num, out_tokens, out_flags);
  return cudaGetLastError();
}

}  // namespace sv
