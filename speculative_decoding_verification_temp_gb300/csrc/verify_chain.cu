// Chain verification (rows 16-byte aligned, no row filters, gamma <= 31) as
// two stream-ordered kernels.  No CTA waits on another CTA's progress except
// at the cluster barriers of one sequence's cluster.
//
//  1. rows kernel (chain_rows.cu), the HBM stream.  Every logit row of the
//     batch - the gamma + 1 target rows and the gamma draft rows of each
//     sequence - is cut into 32 KB chunks, streamed once through shared memory
//     by bulk asynchronous copies, and reduced to one 64-bit record per warp
//     per chunk: (max, sum of 2^((z - max) k)) of a sampling row,
//     k = log2(e) / T, or (finite max, lowest index + 1) of a greedy row.
//  2. draw kernel (this file), one cluster of C CTAs per sequence.  Every CTA
//     of the cluster merges the sequence's records into softmax normalisers
//     (or argmaxes), runs the acceptance tests of all gamma positions at once
//     (u < min(1, p/q), one lane each, Philox uniforms) and finds the first
//     rejection j with a ballot: the same deterministic arithmetic in every
//     CTA, so they agree without exchanging anything.  A one-hot draw needs
//     no weights and CTA 0 writes the outputs.  Otherwise CTA r sums the draw
//     weights ([p_j - q_j]_+ for a correction, p_gamma for the bonus) over
//     its 1/C share of the 256-entry steps, the step totals are gathered into
//     every CTA through distributed shared memory, and each CTA finds the step
//     holding u * W by a double-float prefix and scans it; CTA 0 writes the
//     outputs.  A draw within 1e-6 W of a CDF boundary, closer than the
//     single-precision error of the sums, is redrawn by the same cluster in
//     double-float arithmetic: per-CTA double-float step sums, the exact
//     normaliser ratio from the gathered shares, a double-float search in
//     CTA 0.
//
// Exponent arithmetic: 2^((z - m) k) with z - m computed exactly (one rounding
// in the product), in the records, the merge, the acceptance test and the draw
// alike, so the normalisers and the draw weights share their scale.
#include <algorithm>
#include <mutex>

#include "ops.cuh"
#include "precise_row.cuh"

namespace sv {

cudaError_t launch_chain_rows(const Params &P, int esize, size_t smem, cudaStream_t stream,
                              bool pdl);

namespace {

constexpr int kDWarps = 4;                   // draw kernel
constexpr int kDThreads = kDWarps * 32;
constexpr int kDrawCluster = 4;              // CTAs per sequence (fewer when the row is short)
constexpr int kDrawRecords = 2048;           // records a draw CTA stages in shared memory
constexpr int kPWarps = 8;                   // precise kernel
constexpr int kPThreads = kPWarps * 32;
constexpr int kPreciseCluster = 16;          // CTAs per queued draw (fewer when it cannot run)
constexpr int kPreciseGrid = 32;             // clusters of the precise kernel (queued draws stride)
constexpr int kStep = 256;  // entries per draw-search step
constexpr int kCMaxGamma = 31;
constexpr int kCMaxRows = 2 * kCMaxGamma + 1;
constexpr uint32_t kNoIndex = 0x3FFFFFFFu;  // record index: no finite entry
constexpr uint32_t kBadBit = 0x80000000u;   // record index bit: NaN or +inf seen

// Double-float helpers (FP32 operations only: GB300's FP64 rate is far below
// its FP32 rate).
__device__ __forceinline__ Df df_shfl_xor(Df a, int off) {
  return Df{__shfl_xor_sync(0xFFFFFFFFu, a.hi, off), __shfl_xor_sync(0xFFFFFFFFu, a.lo, off)};
}
__device__ __forceinline__ Df df_shfl_up(Df a, int off) {
  return Df{__shfl_up_sync(0xFFFFFFFFu, a.hi, off), __shfl_up_sync(0xFFFFFFFFu, a.lo, off)};
}
__device__ __forceinline__ Df df_shfl(Df a, int src) {
  return Df{__shfl_sync(0xFFFFFFFFu, a.hi, src), __shfl_sync(0xFFFFFFFFu, a.lo, src)};
}
__device__ __forceinline__ Df df_warp_sum(Df a) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) a = df_add(a, df_shfl_xor(a, off));
  return a;
}
// a > b for normalised double-floats
__device__ __forceinline__ bool df_gt(Df a, Df b) { return df_sub(a, b).hi > 0.f; }

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialisation may start while the previous kernel in the stream finishes;
// it waits here until that kernel's memory operations are visible.  (A no-op
// for a kernel launched without the attribute.)
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
// Lets the next kernel in the stream start launching its CTAs.
__device__ __forceinline__ void launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Barrier over the draw kernel's CTA (named barrier 1, all kDThreads threads).
__device__ __forceinline__ void wsync() { asm volatile("bar.sync 1, %0;" ::"n"(kDThreads) : "memory"); }

// ---------------------------------------------------------------------------
// 1. rows kernel: chain_rows.cu
// ---------------------------------------------------------------------------

// Policy of a row: greedy (argmax) or sampling with k = log2(e) / T.
__device__ __forceinline__ bool row_is_arg(float T) { return !(T > 0.f) || T == INFINITY; }

template <typename TE>
__device__ __forceinline__ void load_vec(const TE *s, float z[8]);
template <>
__device__ __forceinline__ void load_vec<uint16_t>(const uint16_t *s, float z[8]) {
  const uint4 w = *reinterpret_cast<const uint4 *>(s);
  const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    z[2 * i] = __uint_as_float(ws[i] << 16);
    z[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
  }
}
template <>
__device__ __forceinline__ void load_vec<float>(const float *s, float z[8]) {
  const float4 a = *reinterpret_cast<const float4 *>(s);
  const float4 b = *reinterpret_cast<const float4 *>(s + 4);
  z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
  z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
}

// ---------------------------------------------------------------------------
// 2. draw kernel: the decision
// ---------------------------------------------------------------------------

// 2^((z - m) k): the exponent form every step of the chain path uses.
__device__ __forceinline__ float pexp(float z, float m, float k) {
  return fast_exp2(__fmul_rn(__fsub_rn(z, m), k));
}

// Probability of entry v with logit z under a row descriptor.
// kF: the row may carry a filter threshold (calls with a row filter).
template <bool kF = true>
__device__ __forceinline__ float pprob(const RowDesc &d, float z, int v) {
  if (d.onehot) return v == d.a ? 1.f : 0.f;
  if (kF && !(z >= d.thr)) return 0.f;  // below a filter's threshold
  return pexp(z, d.m, d.k) * d.invS;
}

// Descriptor of a row from its merged record (one lane): greedy rows
// (temperature 0) are one-hot at their argmax, sampling rows carry
// (max, k, 1 / S); rows whose statistics are not finite are one-hot at the
// finite argmax, which the caller fills in.
__device__ __forceinline__ RowDesc row_desc(unsigned long long rec, bool arg, bool tbad, float kk,
                                            int V) {
  const float x = __uint_as_float(static_cast<uint32_t>(rec));
  const uint32_t y = static_cast<uint32_t>(rec >> 32);
  RowDesc d;
  d.thr = -INFINITY;
  d.flags = 0u;
  d.m = 0.f;
  d.k = d.nmk = d.invS = 0.f;
  d.a = 0;
  if (arg) {
    const uint32_t idx = (y & ~kBadBit) - 1u;
    const bool none = rec == 0ull || idx >= static_cast<uint32_t>(V);
    d.onehot = 1;
    d.a = none ? 0 : static_cast<int>(idx);
    if (tbad || (y >> 31) || none) d.flags = SPEC_FLAG_NONFINITE;
    return d;
  }
  const float S = __uint_as_float(y);
  const bool bad = rec == 0ull || S != S || x == INFINITY || !(x > -INFINITY) || !(S > 0.f) ||
                   S == INFINITY;
  if (bad) {
    d.onehot = 1;
    d.flags = SPEC_FLAG_NONFINITE;
  } else {
    d.onehot = 0;
    d.k = kk;
    d.m = x;
    d.nmk = -x * kk;
    d.invS = 1.f / S;
  }
  return d;
}

__device__ __forceinline__ RowDesc shfl_desc(const RowDesc &d, int src) {
  RowDesc o;
  o.onehot = __shfl_sync(0xFFFFFFFFu, d.onehot, src);
  o.a = __shfl_sync(0xFFFFFFFFu, d.a, src);
  o.k = __shfl_sync(0xFFFFFFFFu, d.k, src);
  o.nmk = __shfl_sync(0xFFFFFFFFu, d.nmk, src);
  o.invS = __shfl_sync(0xFFFFFFFFu, d.invS, src);
  o.thr = __shfl_sync(0xFFFFFFFFu, d.thr, src);
  o.flags = __shfl_sync(0xFFFFFFFFu, d.flags, src);
  o.m = __shfl_sync(0xFFFFFFFFu, d.m, src);
  return o;
}


// Finite argmax of a whole row (one warp; rows whose sampling statistics were
// not finite, a rare path).
template <typename TE>
__device__ int warp_finite_argmax(const TE *g, int V) {
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
    argmax_merge(bv, bi, v2, i2);
  }
  return bi == INT_MAX ? 0 : bi;
}

// Row r of sequence seq (target rows 0..gamma, then the gamma draft rows).
template <typename TE>
__device__ __forceinline__ const TE *chain_row(const Params &P, int seq, int r) {
  const bool draft = r > P.gamma;
  const long long row = draft ? static_cast<long long>(seq) * P.gamma + (r - P.gamma - 1)
                              : static_cast<long long>(seq) * (P.gamma + 1) + r;
  return static_cast<const TE *>(
      row_ptr(draft ? P.draft : P.target, row, draft ? P.ld_d : P.ld_t, sizeof(TE)));
}


// Outputs of a finished sequence and the unit record the residual output
// reads (one thread).
__device__ void write_outputs(const Params &P, int s, const PassSeq &ps, int token, double W,
                              int near) {
  const long long obase = static_cast<long long>(s) * (P.gamma + 1);
  const long long unit = obase + ps.j;
  for (int i = 0; i <= P.gamma; ++i) {
    int v = -1;
    if (i < ps.j) v = __ldg(P.tokens + static_cast<long long>(s) * P.gamma + i);
    else if (i == ps.j) v = token;
    P.out_tokens[obase + i] = v;
  }
  P.out_num[s] = ps.j;
  if (P.out_flags) P.out_flags[s] = ps.flags;
  UnitOut o;
  o.next = -1;
  o.token = token;
  o.flags = ps.flags;
  o.near = near;
  P.outs[unit] = o;
  UnitStats st;
  st.p = ps.dp;
  st.q = ps.dq;
  st.c = ps.residual ? 1.f : 0.f;
  st.total = static_cast<float>(W);
  st.kind = ps.kind;
  st.node = ps.j;
  st.n_res = ps.residual;
  st.pad = 0;
  P.stats[unit] = st;
  P.final_unit[s] = static_cast<int>(unit);
}

// The merged record of row r of sequence (or tree) seq (one warp; the value in
// every lane) from the row's R records at `rec` (global memory, or a
// shared-memory copy): the rows kernel stored all of them before this kernel.
// A chain's rows are its gamma + 1 target rows, then its draft rows; a tree's
// its N target rows, then its N draft rows.
__device__ unsigned long long merge_row(const Params &P, int seq, int r,
                                        const unsigned long long *rec, bool shared) {
  const int lane = threadIdx.x & 31;
  const bool draft = P.mode == kModeTree ? r >= P.ups : r > P.gamma;
  const float T = __ldg((draft ? P.Tq : P.Tp) + seq);
  const bool arg = row_is_arg(T);
  const float k = arg ? 0.f : kLog2e / T;
  const int R = P.cpr * kChainRecordsPerChunk;
  float m = -INFINITY, S = 0.f, bv = -INFINITY;
  uint32_t bi = kNoIndex;
  int bad = 0;
  for (int x0 = lane; x0 < R; x0 += 4 * 32) {
    unsigned long long b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i)
      b[i] = x0 + i * 32 < R ? (shared ? rec[x0 + i * 32] : __ldcg(rec + x0 + i * 32)) : 0ull;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (x0 + i * 32 >= R) continue;
      const float qx = __uint_as_float(static_cast<uint32_t>(b[i]));
      const uint32_t qy = static_cast<uint32_t>(b[i] >> 32);
      if (arg) {
        bad |= static_cast<int>(qy >> 31);
        const uint32_t idx = (qy & ~kBadBit) - 1u;
        if (qx > bv || (qx == bv && idx < bi)) {
          bv = qx;
          bi = idx;
        }
      } else {
        const float qs = __uint_as_float(qy);
        if (qs != qs || qx == INFINITY) bad = 1;
        else online_merge(m, S, qx, qs, k);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, off);
    const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, off);
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
    const uint32_t i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
    bad |= __shfl_xor_sync(0xFFFFFFFFu, bad, off);
    if (!arg) online_merge(m, S, m2, S2, k);
    if (v2 > bv || (v2 == bv && i2 < bi)) {
      bv = v2;
      bi = i2;
    }
  }
  // the row's record, in the chunk records' format (never zero)
  uint32_t lo, hi;
  if (arg) {
    lo = __float_as_uint(bv);
    hi = (bi + 1u) | (bad ? kBadBit : 0u);
  } else {
    lo = __float_as_uint(m);
    hi = bad ? 0x7FC00000u : __float_as_uint(S);
  }
  return static_cast<unsigned long long>(lo) | (static_cast<unsigned long long>(hi) << 32);
}

// What the decision of sequence seq reads from the inputs alone (one warp,
// lane i: draft position i), loaded before the rows kernel has finished.
struct DecideIn {
  float Tp, Tq;
  int x;         // draft token of position i
  float zp, zq;  // logits of x in target row i and draft row i (0 when x is not valid)
  float ua, ud;  // acceptance and draw uniforms of position i
};

template <typename TE>
__device__ DecideIn decide_inputs(const Params &P, int seq) {
  const int i = threadIdx.x & 31;
  const int gamma = P.gamma, V = P.V;
  DecideIn in;
  in.Tp = __ldg(P.Tp + seq);
  in.Tq = __ldg(P.Tq + seq);
  in.x = i < gamma ? __ldg(P.tokens + static_cast<long long>(seq) * gamma + i) : -1;
  const bool valid = i < gamma && in.x >= 0 && in.x < V;
  in.zp = valid ? to_f32(chain_row<TE>(P, seq, i)[in.x]) : 0.f;
  in.zq = valid ? to_f32(chain_row<TE>(P, seq, gamma + 1 + i)[in.x]) : 0.f;
  in.ua = i < gamma ? unit_uniform(P, seq, i, 0) : 0.f;
  in.ud = i <= gamma ? unit_uniform(P, seq, i, 1) : 0.f;
  return in;
}

// Decide sequence seq from its rows' records (one warp): the acceptance
// tests, the first rejection j, and the draw's description in `out` (lane 0).
// A one-hot draw needs no weights: the writer CTA writes its outputs.
template <typename TE, bool kF>
__device__ void decide_seq(const Params &P, int seq, const unsigned long long *rr,
                           const DecideIn &in, bool writer, PassSeq &out) {
  const int lane = threadIdx.x & 31;
  const int gamma = P.gamma, V = P.V;
  const float Tp = in.Tp, Tq = in.Tq;
  const bool p_arg = row_is_arg(Tp), q_arg = row_is_arg(Tq);
  const bool tp_bad = !(Tp >= 0.f) || Tp == INFINITY, tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  const float kp = p_arg ? 0.f : kLog2e / Tp, kq = q_arg ? 0.f : kLog2e / Tq;
  // lane i holds target row i (i <= gamma) and draft row gamma + 1 + i (i < gamma)
  const int i = lane;
  RowDesc dp = row_desc(i <= gamma ? rr[i] : 0ull, p_arg, tp_bad, kp, V);
  // a greedy target never reads q (its draft rows have no records): a one-hot
  // stand-in
  RowDesc dq = row_desc(i < gamma && !p_arg ? rr[gamma + 1 + i] : 0ull, q_arg || p_arg, tq_bad, kq, V);
  if (p_arg) dq.flags = 0u;
  if (kF) {
    // filtered rows: the filter kernel's threshold and kept normaliser
    const long long rb = static_cast<long long>(seq) * (2 * gamma + 1);
    const float2 fp = i <= gamma ? __ldcg(P.frec + rb + i) : make_float2(-INFINITY, 0.f);
    const float2 fq = i < gamma ? __ldcg(P.frec + rb + gamma + 1 + i) : make_float2(-INFINITY, 0.f);
    if (!dp.onehot && fp.y > 0.f) {
      dp.thr = fp.x;
      dp.invS = 1.f / fp.y;
    }
    if (!dq.onehot && fq.y > 0.f) {
      dq.thr = fq.x;
      dq.invS = 1.f / fq.y;
    }
  }
  // rows whose sampling statistics were not finite: the finite argmax (rare)
  unsigned need = __ballot_sync(0xFFFFFFFFu, i <= gamma && !p_arg && dp.onehot);
  while (need) {
    const int src = __ffs(need) - 1;
    need &= need - 1;
    const int a = warp_finite_argmax<TE>(chain_row<TE>(P, seq, src), V);
    if (lane == src) dp.a = a;
  }
  need = __ballot_sync(0xFFFFFFFFu, i < gamma && !p_arg && !q_arg && dq.onehot);
  while (need) {
    const int src = __ffs(need) - 1;
    need &= need - 1;
    const int a = warp_finite_argmax<TE>(chain_row<TE>(P, seq, gamma + 1 + src), V);
    if (lane == src) dq.a = a;
  }
  // acceptance tests, one lane per draft position
  uint32_t f = 0u;
  bool reject = true;
  if (i < gamma) {
    const int x = in.x;
    f = dp.flags;
    const bool valid = x >= 0 && x < V;
    if (!valid) f |= SPEC_FLAG_BAD_TOKEN;
    if (dp.onehot) {
      reject = !(valid && x == dp.a);
    } else {
      f |= dq.flags;
      if (valid) {
        const float px = pprob<kF>(dp, in.zp, x);
        const float qx = pprob<kF>(dq, dq.onehot ? 0.f : in.zq, x);
        if (!(qx > 0.f)) {
          f |= SPEC_FLAG_ZERO_Q;
        } else {
          reject = !(in.ua < fminf(1.f, px / qx));
        }
      }
    }
  }
  const unsigned rej = __ballot_sync(0xFFFFFFFFu, reject && i < gamma);
  const int j = rej ? __ffs(rej) - 1 : gamma;
  const float u_draw = __shfl_sync(0xFFFFFFFFu, in.ud, j);
  uint32_t fo = warp_or(i < j ? f : 0u);
  fo |= __shfl_sync(0xFFFFFFFFu, i < gamma ? f : dp.flags, j);  // position j's flags
  const RowDesc djp = shfl_desc(dp, j);
  const RowDesc djq = shfl_desc(dq, j);
  if (lane == 0 && __ldcg(P.err)) {
    // a bounded wait of the rows kernel gave up: the documented fallback, no
    // accepted drafts and no tokens
    if (writer) {
      const long long obase = static_cast<long long>(seq) * (gamma + 1);
      for (int x = 0; x <= gamma; ++x) P.out_tokens[obase + x] = -1;
      P.out_num[seq] = 0;
      if (P.out_flags) P.out_flags[seq] = SPEC_FLAG_TIMEOUT;
      P.final_unit[seq] = -1;
    }
    PassSeq ps = {};
    ps.draw = 0;
    out = ps;
    return;
  }
  if (lane == 0) {
    PassSeq ps;
    ps.dp = djp;
    ps.residual = j < gamma ? 1 : 0;
    if (ps.residual) {
      ps.dq = djq;
    } else {
      ps.dq = djp;
      ps.dq.onehot = 1;
      ps.dq.a = 0;
    }
    ps.j = j;
    ps.flags = fo;
    ps.W = 0.f;
    ps.u = u_draw;
    ps.kind = j < gamma ? 2 : 0;
    ps.draw = 1;
    if (ps.dp.onehot) {  // the token needs no draw: finish the sequence here
      ps.kind = j < gamma ? 1 : 0;
      ps.residual = 0;
      ps.draw = 0;
      ps.u = 0.f;
      if (writer) write_outputs(P, seq, ps, ps.dp.a, 0.0, 0);
    }
    out = ps;
  }
}

// ---------------------------------------------------------------------------
// 2b. filter kernel: top-k / top-p / min-p thresholds of filtered rows
// ---------------------------------------------------------------------------

constexpr int kFThreads = 256;
constexpr int kFWarps = kFThreads / 32;
constexpr int kFMaxBlocks = 4096;  // 512-entry blocks per row (V <= 2,097,152)

struct FilterShared {
  unsigned long long rec;  // the row's merged record
  int hist[256];
  unsigned long long mhist[256];
  uint32_t prefix;
  int kk;
  int found;
  unsigned long long need;
  unsigned long long wtot[kFWarps];
  float wsum[kFWarps];
  int wcnt[kFWarps];
  int ncand;
  uint32_t bkey[kFMaxBlocks];  // block-max order keys
  int cand[kFMaxBlocks];       // candidate blocks, ascending
};

// Scan of a 256-bin histogram from the top digit (warp 0): the digit at which
// the running sum reaches `need`, and what is left of `need` inside it.  The
// histogram total goes to `total`.
template <typename T>
__device__ __forceinline__ void scan_top(const T *hist, T need, int &digit, T &left, T &total) {
  const int lane = threadIdx.x & 31;
  // lane l owns digits 255 - 8 l - j, j = 0..7 (descending values)
  T cnt[8];
  T s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    cnt[j] = hist[255 - 8 * lane - j];
    s += cnt[j];
  }
  T incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += t;
  }
  total = __shfl_sync(0xFFFFFFFFu, incl, 31);
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, incl >= need);
  const int first = bal ? __ffs(bal) - 1 : 31;
  int d = 0;
  T l = 0;
  if (lane == first) {
    T acc = incl - s;
    d = 255 - 8 * lane - 7;
    l = need - (acc < need ? acc : need);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (acc + cnt[j] >= need) {
        d = 255 - 8 * lane - j;
        l = need - acc;
        break;
      }
      acc += cnt[j];
    }
  }
  digit = __shfl_sync(0xFFFFFFFFu, d, first);
  left = __shfl_sync(0xFFFFFFFFu, l, first);
}

// Order key of the kk-th largest of the n keys item(i, key) yields (false:
// no key), 8 bits a round from the top of KB-bit keys; false when fewer
// than kk keys exist.  The whole CTA calls it.
template <int KB, typename F>
__device__ bool kth_key(FilterShared &sh, int n, int kk, F item, uint32_t &out) {
  const int tid = threadIdx.x;
  if (tid == 0) {
    sh.prefix = 0u;
    sh.kk = kk;
    sh.found = 1;
  }
  for (int round = 0; round < KB / 8; ++round) {
    const int shift = KB - 8 * (round + 1);
    for (int i = tid; i < 256; i += kFThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t hmask = round == 0 ? 0u : (0xFFFFFFFFu << (KB - 8 * round));
    const uint32_t want = round == 0 ? 0u : (sh.prefix << (KB - 8 * round));
    for (int i = tid; i < n; i += kFThreads) {
      uint32_t key;
      if (item(i, key) && (key & hmask) == want) atomicAdd(&sh.hist[(key >> shift) & 255u], 1);
    }
    __syncthreads();
    if (tid < 32) {
      int d, left, total;
      scan_top<int>(sh.hist, sh.kk, d, left, total);
      if (tid == 0) {
        if (round == 0 && total < sh.kk) sh.found = 0;
        sh.prefix = (sh.prefix << 8) | static_cast<uint32_t>(d);
        sh.kk = left;
      }
    }
    __syncthreads();
    if (!sh.found) return false;
  }
  out = sh.prefix;
  return true;
}

// Order key of a logit held as a float (for bf16 rows, the key of its bf16
// bits).
template <typename TE>
__device__ __forceinline__ uint32_t zkey(float z) {
  return sizeof(TE) == 2 ? order_key(static_cast<uint16_t>(__float_as_uint(z) >> 16))
                         : order_key(z);
}

// Per-warp regions of the compact candidate list (the block-key array's
// storage, free once the candidate blocks are known).
constexpr int kFCap = kFMaxBlocks / kFWarps;

__device__ __forceinline__ const float *flist(const FilterShared &sh) {
  return reinterpret_cast<const float *>(sh.bkey);
}

// Entry i of the compact list (warp region i / kFCap): false past the
// region's count.
__device__ __forceinline__ bool list_entry(const FilterShared &sh, int i, float &z) {
  const int w = i / kFCap;
  if (i - w * kFCap >= sh.wcnt[w]) return false;
  z = flist(sh)[i];
  return true;
}

// mass_key over the compact list's entries at or above lo.
template <typename TE>
__device__ bool mass_list(FilterShared &sh, float lo, float m, float k, unsigned long long need,
                          uint32_t &out) {
  constexpr int KB = sizeof(TE) == 2 ? 16 : 32;
  const int tid = threadIdx.x, lane = tid & 31;
  if (tid == 0) {
    sh.prefix = 0u;
    sh.need = need;
    sh.found = 1;
  }
  for (int round = 0; round < KB / 8; ++round) {
    const int shift = KB - 8 * (round + 1);
    for (int i = tid; i < 256; i += kFThreads) sh.mhist[i] = 0ull;
    __syncthreads();
    const uint32_t hmask = round == 0 ? 0u : (0xFFFFFFFFu << (KB - 8 * round));
    const uint32_t want = round == 0 ? 0u : (sh.prefix << (KB - 8 * round));
    for (int i0 = tid - lane; i0 < kFWarps * kFCap; i0 += kFThreads) {  // warp-uniform
      float z = 0.f;
      const bool have = list_entry(sh, i0 + lane, z);
      const uint32_t key = zkey<TE>(z);
      const bool in = have && z >= lo && (key & hmask) == want;
      warp_hist_mass(sh.mhist, in ? static_cast<int>((key >> shift) & 255u) : -1,
                     in ? mass_fixed(z, m, k) : 0ull);
    }
    __syncthreads();
    if (tid < 32) {
      int d;
      unsigned long long left, total;
      scan_top<unsigned long long>(sh.mhist, sh.need, d, left, total);
      if (tid == 0) {
        if (round == 0 && total < sh.need) sh.found = 0;
        sh.prefix = (sh.prefix << 8) | static_cast<uint32_t>(d);
        sh.need = left;
      }
    }
    __syncthreads();
    if (!sh.found) return false;
  }
  out = sh.prefix;
  return true;
}

template <typename TE>
__device__ __forceinline__ float key_value(uint32_t k) {
  return sizeof(TE) == 2 ? key_value_bf16(k) : key_value_f32(k);
}

// One pass over the candidate blocks' entries, 8 at a time (64 groups a
// block), four groups of a thread in flight: f(z[8], v0, ok) for every group,
// v0 the vocabulary index of z[0] (entries at or past V read -inf), ok false
// for a thread past the last group.  Every lane of a warp calls f the same
// number of times, so f may use warp-collective operations.
template <typename TE, typename F>
__device__ void for_groups(const FilterShared &sh, const TE *g, int V, int ngroups, F f) {
  const int lane = threadIdx.x & 31;
  for (int jw = threadIdx.x - lane; jw < ngroups; jw += 4 * kFThreads) {
    float z[4][8];
    int v0[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int j = jw + lane + q * kFThreads;
      const bool ok = j < ngroups;
      v0[q] = ok ? sh.cand[j >> 6] * 512 + (j & 63) * 8 : V;
      hp_load8<TE>(g, v0[q], ok ? V : 0, true, z[q]);
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (jw + q * kFThreads >= ngroups) break;  // warp-uniform
      f(z[q], v0[q], jw + lane + q * kFThreads < ngroups);
    }
  }
}

// kth_key over the candidate entries (count histograms).
template <typename TE>
__device__ bool kth_entry(FilterShared &sh, const TE *g, int V, int ngroups, int kk,
                          uint32_t &out) {
  constexpr int KB = sizeof(TE) == 2 ? 16 : 32;
  const int tid = threadIdx.x;
  if (tid == 0) {
    sh.prefix = 0u;
    sh.kk = kk;
    sh.found = 1;
  }
  for (int round = 0; round < KB / 8; ++round) {
    const int shift = KB - 8 * (round + 1);
    for (int i = tid; i < 256; i += kFThreads) sh.hist[i] = 0;
    __syncthreads();
    const uint32_t hmask = round == 0 ? 0u : (0xFFFFFFFFu << (KB - 8 * round));
    const uint32_t want = round == 0 ? 0u : (sh.prefix << (KB - 8 * round));
    for_groups<TE>(sh, g, V, ngroups, [&](const float *z, int v0, bool ok) {
      if (!ok) return;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t key = zkey<TE>(z[e]);
        if (v0 + e < V && (key & hmask) == want) atomicAdd(&sh.hist[(key >> shift) & 255u], 1);
      }
    });
    __syncthreads();
    if (tid < 32) {
      int d, left, total;
      scan_top<int>(sh.hist, sh.kk, d, left, total);
      if (tid == 0) {
        if (round == 0 && total < sh.kk) sh.found = 0;
        sh.prefix = (sh.prefix << 8) | static_cast<uint32_t>(d);
        sh.kk = left;
      }
    }
    __syncthreads();
    if (!sh.found) return false;
  }
  out = sh.prefix;
  return true;
}

// mass_key over the candidate entries at or above lo.
template <typename TE>
__device__ bool mass_entry(FilterShared &sh, const TE *g, int V, int ngroups, float lo, float m,
                           float k, unsigned long long need, uint32_t &out) {
  constexpr int KB = sizeof(TE) == 2 ? 16 : 32;
  const int tid = threadIdx.x;
  if (tid == 0) {
    sh.prefix = 0u;
    sh.need = need;
    sh.found = 1;
  }
  for (int round = 0; round < KB / 8; ++round) {
    const int shift = KB - 8 * (round + 1);
    for (int i = tid; i < 256; i += kFThreads) sh.mhist[i] = 0ull;
    __syncthreads();
    const uint32_t hmask = round == 0 ? 0u : (0xFFFFFFFFu << (KB - 8 * round));
    const uint32_t want = round == 0 ? 0u : (sh.prefix << (KB - 8 * round));
    for_groups<TE>(sh, g, V, ngroups, [&](const float *z, int v0, bool ok) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const uint32_t key = zkey<TE>(z[e]);
        const bool in = ok && v0 + e < V && z[e] >= lo && (key & hmask) == want;
        warp_hist_mass(sh.mhist, in ? static_cast<int>((key >> shift) & 255u) : -1,
                       in ? mass_fixed(z[e], m, k) : 0ull);
      }
    });
    __syncthreads();
    if (tid < 32) {
      int d;
      unsigned long long left, total;
      scan_top<unsigned long long>(sh.mhist, sh.need, d, left, total);
      if (tid == 0) {
        if (round == 0 && total < sh.need) sh.found = 0;
        sh.prefix = (sh.prefix << 8) | static_cast<uint32_t>(d);
        sh.need = left;
      }
    }
    __syncthreads();
    if (!sh.found) return false;
  }
  out = sh.prefix;
  return true;
}

// One CTA per row (grid: nseq (2 gamma + 1)), after the rows kernel.  For a
// sampled row with a filter it writes frec[row] = (threshold, S over the kept
// entries), else (-inf, 0).  The filters, in order: top-k on the logits (every
// entry tied with the k-th largest kept), top-p on the distribution after
// temperature and top-k (the smallest prefix of the descending values whose
// mass reaches top_p of the kept mass, ties kept), min-p (p >= min_p max p,
// i.e. z >= max + T ln min_p).  The kept set is {z >= max(thresholds)}.
//
// Only 512-entry blocks that can hold a kept entry are read: a lower bound L
// of the final threshold selects them (block max >= L).  L is the k-th
// largest block maximum (at most the k-th largest entry), or the min-p
// boundary, or both; with top-p and no top-k, the top-p total needs either
// every entry (no min-p: L = -inf) or the row statistics (with min-p: the
// total is the single-precision S of the row).
template <typename TE>
__global__ void __launch_bounds__(kFThreads) chain_filter_kernel(const Params P) {
  __shared__ FilterShared sh;
  constexpr int KB = sizeof(TE) == 2 ? 16 : 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rps = 2 * P.gamma + 1;
  const int rowid = static_cast<int>(blockIdx.x);
  const int seq = rowid / rps, r = rowid - seq * rps;
  const bool draft = r > P.gamma;
  launch_dependents();
  const float T = __ldg((draft ? P.Tq : P.Tp) + seq);
  const int *kpa = draft ? P.kq : P.kp;
  const float *ppa = draft ? P.pq : P.pp;
  const float *mpa = draft ? P.mq : P.mp;
  const int V = P.V, nblk = P.nblk;
  int kk = kpa ? __ldg(kpa + seq) : 0;
  if (kk <= 0 || kk >= V) kk = 0;
  const float tpr = ppa ? __ldg(ppa + seq) : 1.f;
  const float mpr = mpa ? __ldg(mpa + seq) : 0.f;
  const bool topp = tpr < 1.f;  // NaN: off
  const bool minp = mpr > 0.f;  // NaN: off
  grid_dependency_wait();  // the rows kernel's records and block maxima
  // greedy rows, and the draft rows of a greedy target (never read), take no
  // filter
  if (row_is_arg(T) || (draft && row_is_arg(__ldg(P.Tp + seq))) || (!kk && !topp && !minp)) {
    if (tid == 0) P.frec[rowid] = make_float2(-INFINITY, 0.f);
    return;
  }
  const TE *g = chain_row<TE>(P, seq, r);
  if (warp == 0) {
    const int R = P.cpr * kChainRecordsPerChunk;
    const unsigned long long rec =
        merge_row(P, seq, r, P.srec + static_cast<long long>(rowid) * R, false);
    if (lane == 0) sh.rec = rec;
  }
  __syncthreads();
  const float m = __uint_as_float(static_cast<uint32_t>(sh.rec));
  const float Srow = __uint_as_float(static_cast<uint32_t>(sh.rec >> 32));
  if (!(m > -INFINITY) || m == INFINITY || !(Srow > 0.f) || Srow == INFINITY) {
    // statistics that are not finite: the draw kernel takes the one-hot
    if (tid == 0) P.frec[rowid] = make_float2(-INFINITY, 0.f);
    return;
  }
  const float k = kLog2e / T;
  const float Lm = minp ? m + T * logf(fminf(mpr, 1.f)) : -INFINITY;
  // 1. the lower bound L and the candidate blocks
  const TE *bm = static_cast<const TE *>(P.bmax) + static_cast<long long>(rowid) * nblk;
  float L = -INFINITY;
  if (kk) {
    for (int b = tid; b < nblk; b += kFThreads) sh.bkey[b] = order_key(bm[b]);
    __syncthreads();
    uint32_t key;
    const bool ok = kth_key<KB>(sh, nblk, kk, [&](int i, uint32_t &kx) {
      kx = sh.bkey[i];
      return true;
    }, key);
    L = ok ? key_value<TE>(key) : -INFINITY;
    if (!topp) L = fmaxf(L, Lm);
  } else if (minp) {
    L = Lm;
  }
  {
    int base = 0;
    for (int b0 = 0; b0 < nblk; b0 += kFThreads) {
      const int b = b0 + tid;
      const bool c = b < nblk && to_f32(bm[b]) >= L;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, c);
      if (lane == 0) sh.wcnt[warp] = __popc(bal);
      __syncthreads();
      int off = base;
      for (int x = 0; x < warp; ++x) off += sh.wcnt[x];
      if (c) sh.cand[off + __popc(bal & ((1u << lane) - 1u))] = b;
      int tot = 0;
      for (int x = 0; x < kFWarps; ++x) tot += sh.wcnt[x];
      base += tot;
      __syncthreads();
    }
    if (tid == 0) sh.ncand = base;
    __syncthreads();
  }
  const int ngroups = sh.ncand * 64;
  // 2. the candidate entries (z >= L) into per-warp regions of a compact
  // list in shared memory, in a fixed order; the global passes below run only
  // when a region overflows
  {
    float *list = reinterpret_cast<float *>(sh.bkey);
    int wbase = 0;
    for_groups<TE>(sh, g, V, ngroups, [&](const float *z, int v0, bool ok) {
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const bool in = ok && v0 + e < V && z[e] >= L;
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, in);
        const int pos = wbase + __popc(bal & ((1u << lane) - 1u));
        if (in && pos < kFCap) list[warp * kFCap + pos] = z[e];
        wbase += __popc(bal);
      }
    });
    if (lane == 0) sh.wcnt[warp] = wbase;
    __syncthreads();
  }
  bool over = false;
  for (int x = 0; x < kFWarps; ++x) over |= sh.wcnt[x] > kFCap;
  if (!over) {
    float tk = -INFINITY;
    if (kk) {
      uint32_t key;
      const bool ok = kth_key<KB>(sh, kFWarps * kFCap, kk, [&](int i, uint32_t &kx) {
        float z;
        if (!list_entry(sh, i, z)) return false;
        kx = zkey<TE>(z);
        return true;
      }, key);
      tk = ok ? key_value<TE>(key) : -INFINITY;
    }
    float tpv = -INFINITY;
    if (topp) {
      unsigned long long total;
      if (kk) {
        unsigned long long t = 0ull;
        for (int i = tid; i < kFWarps * kFCap; i += kFThreads) {
          float z;
          if (list_entry(sh, i, z) && z >= tk) t += mass_fixed(z, m, k);
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
        if (lane == 0) sh.wtot[warp] = t;
        __syncthreads();
        total = 0ull;
        for (int x = 0; x < kFWarps; ++x) total += sh.wtot[x];
        __syncthreads();
      } else {
        total = __float2ull_rn(Srow * kMassScale);
      }
      const float tp = fmaxf(tpr, 0.f);
      const double t = static_cast<double>(tp) * static_cast<double>(total);
      unsigned long long need = static_cast<unsigned long long>(t);
      if (static_cast<double>(need) < t) ++need;
      if (need == 0ull) need = 1ull;
      uint32_t key;
      tpv = mass_list<TE>(sh, fmaxf(tk, Lm), m, k, need, key) ? key_value<TE>(key) : -INFINITY;
    }
    const float thr = fmaxf(fmaxf(tk, tpv), Lm);
    float s = 0.f;
    for (int i = tid; i < kFWarps * kFCap; i += kFThreads) {
      float z;
      if (list_entry(sh, i, z) && z >= thr) s += pexp(z, m, k);
    }
    s = warp_sum(s);
    if (lane == 0) sh.wsum[warp] = s;
    __syncthreads();
    if (tid == 0) {
      float S = 0.f;
      for (int x = 0; x < kFWarps; ++x) S += sh.wsum[x];
      P.frec[rowid] = make_float2(thr, S);
    }
    return;
  }
  // 3. top-k: the k-th largest entry (every kept entry is a candidate)
  float tk = -INFINITY;
  if (kk) {
    uint32_t key;
    // not found: fewer than k candidates at or above the min-p boundary, so
    // the top-k boundary lies below it
    tk = kth_entry<TE>(sh, g, V, ngroups, kk, key) ? key_value<TE>(key) : -INFINITY;
  }
  // 4. top-p over the entries at or above the top-k boundary
  float tpv = -INFINITY;
  if (topp) {
    unsigned long long total;
    if (kk || !minp) {
      // every entry of the top-k set is a candidate: the exact total
      unsigned long long t = 0ull;
      for_groups<TE>(sh, g, V, ngroups, [&](const float *z, int v0, bool ok) {
        if (!ok) return;
#pragma unroll
        for (int e = 0; e < 8; ++e)
          if (v0 + e < V && z[e] >= tk) t += mass_fixed(z[e], m, k);
      });
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xFFFFFFFFu, t, off);
      if (lane == 0) sh.wtot[warp] = t;
      __syncthreads();
      total = 0ull;
      for (int x = 0; x < kFWarps; ++x) total += sh.wtot[x];
      __syncthreads();
    } else {
      // top-p and min-p without top-k: the candidates are the min-p set; the
      // total is the row's single-precision S (in the same fixed point)
      total = __float2ull_rn(Srow * kMassScale);
    }
    const float tp = fmaxf(tpr, 0.f);
    const double t = static_cast<double>(tp) * static_cast<double>(total);
    unsigned long long need = static_cast<unsigned long long>(t);
    if (static_cast<double>(need) < t) ++need;  // ceil: the mass must reach top_p
    if (need == 0ull) need = 1ull;               // top_p <= 0 keeps the largest value
    uint32_t key;
    // not found: the top-p boundary lies below the min-p boundary
    tpv = mass_entry<TE>(sh, g, V, ngroups, fmaxf(tk, Lm), m, k, need, key) ? key_value<TE>(key)
                                                                            : -INFINITY;
  }
  // 5. the kept set and its normaliser
  const float thr = fmaxf(fmaxf(tk, tpv), Lm);
  float s = 0.f;
  for_groups<TE>(sh, g, V, ngroups, [&](const float *z, int v0, bool ok) {
    if (!ok) return;
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (v0 + e < V && z[e] >= thr) s += pexp(z[e], m, k);
  });
  s = warp_sum(s);
  if (lane == 0) sh.wsum[warp] = s;
  __syncthreads();
  if (tid == 0) {
    float S = 0.f;
    for (int x = 0; x < kFWarps; ++x) S += sh.wsum[x];
    P.frec[rowid] = make_float2(thr, S);
  }
}

// ---------------------------------------------------------------------------
// 3. draw kernel: the draw weights
// ---------------------------------------------------------------------------

// Eight consecutive logits held as loaded (16 or 32 bytes), converted on use.
template <typename TE>
struct Raw8;
template <>
struct Raw8<uint16_t> {
  uint4 w = make_uint4(0u, 0u, 0u, 0u);
  __device__ __forceinline__ void load(const uint16_t *s) {
    w = *reinterpret_cast<const uint4 *>(s);
  }
  __device__ __forceinline__ void get(float z[8]) const {
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      z[2 * i] = __uint_as_float(ws[i] << 16);
      z[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
    }
  }
};
template <>
struct Raw8<float> {
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f), b = make_float4(0.f, 0.f, 0.f, 0.f);
  __device__ __forceinline__ void load(const float *s) {
    a = *reinterpret_cast<const float4 *>(s);
    b = *reinterpret_cast<const float4 *>(s + 4);
  }
  __device__ __forceinline__ void get(float z[8]) const {
    z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
    z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
  }
};

// Draw weights of the 8 entries from `base` given their logits.  Sampling
// rows without a filter threshold use packed pairs, rounding exactly like
// pprob(); filtered rows take pprob() entry by entry.
template <bool kF>
__device__ __forceinline__ void weights8(const RowDesc &dp, const RowDesc &dq, int residual,
                                         int base, const float zp[8], const float zq[8],
                                         float w[8]) {
  if (!dp.onehot && (!residual || !dq.onehot) &&
      (!kF || (dp.thr == -INFINITY && (!residual || dq.thr == -INFINITY)))) {
    const uint64_t np2 = pack2(-dp.m, -dp.m), kp2 = pack2(dp.k, dp.k),
                   ip2 = pack2(dp.invS, dp.invS);
    const uint64_t nq2 = pack2(-dq.m, -dq.m), kq2 = pack2(dq.k, dq.k),
                   iq2 = pack2(dq.invS, dq.invS);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      const uint64_t p2 = fmul2(ex2_pair(fmul2(fadd2(pack2(zp[e], zp[e + 1]), np2), kp2)), ip2);
      if (residual) {
        const uint64_t q2 =
            fmul2(ex2_pair(fmul2(fadd2(pack2(zq[e], zq[e + 1]), nq2), kq2)), iq2);
        float d0, d1;
        unpack2(fadd2(p2, q2 ^ 0x8000000080000000ull), d0, d1);
        w[e] = fmaxf(d0, 0.f);
        w[e + 1] = fmaxf(d1, 0.f);
      } else {
        unpack2(p2, w[e], w[e + 1]);
      }
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    float x = pprob<kF>(dp, zp[e], base + e);
    if (residual) x = fmaxf(x - pprob<kF>(dq, zq[e], base + e), 0.f);
    w[e] = x;
  }
}

// Draw weights of 8 entries from `base` (entries at or past V are 0).  The
// rows' entry v is at gp[v - off], gq[v - off] (off: the first entry of a
// shared-memory copy of part of the rows, else 0).
template <typename TE, bool kF>
__device__ __forceinline__ void step_weights(const TE *gp, const TE *gq, const RowDesc &dp,
                                             const RowDesc &dq, int residual, int base, int V,
                                             float w[8], int off = 0) {
  float zp[8], zq[8];
  const bool full = base + 8 <= V;
  if (full && !dp.onehot) {
    load_vec<TE>(gp + (base - off), zp);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e)
      zp[e] = (!dp.onehot && base + e < V) ? to_f32(gp[base + e - off]) : 0.f;
  }
  if (residual) {
    if (full && !dq.onehot) {
      load_vec<TE>(gq + (base - off), zq);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        zq[e] = (!dq.onehot && base + e < V) ? to_f32(gq[base + e - off]) : 0.f;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) zq[e] = 0.f;
  }
  weights8<kF>(dp, dq, residual, base, zp, zq, w);  // the same arithmetic as the records
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (base + e >= V) w[e] = 0.f;
}

// Totals of the draw weights of steps [b0, b1) (256 entries each) into
// fst[step] (the NW warps of the CTA, one warp per step; full steps 4 kM
// (bf16) or 2 kM (fp32) per warp at a time with their loads issued before any
// is used).  Entry v of the rows is at gp[v - off], gq[v - off].
template <typename TE, int NW, bool kF, int kM = 1>
__device__ void step_totals(const TE *gp, const TE *gq, const RowDesc &dp, const RowDesc &dq,
                            int residual, int V, int b0, int b1, float *fst,
                            const TE *bmp = nullptr, int off = 0) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // 16 or 32 raw bytes a lane per step and row
  constexpr int kU = (sizeof(TE) == 2 ? 4 : 2) * kM;
  const int nfull = min(b1, V / kStep);
  int st0 = b0 + w;
  if constexpr (!kF) {
    if (!dp.onehot && (!residual || !dq.onehot)) {
      for (; st0 + (kU - 1) * NW < nfull; st0 += NW * kU) {
        Raw8<TE> rp[kU], rq[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int base = (st0 + q * NW) * kStep + lane * 8;
          rp[q].load(gp + (base - off));
          if (residual) rq[q].load(gq + (base - off));
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int base = (st0 + q * NW) * kStep + lane * 8;
          float zp[8], zq[8], x[8];
          rp[q].get(zp);
          rq[q].get(zq);
          weights8<kF>(dp, dq, residual, base, zp, zq, x);
          float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
          sm = warp_sum(sm);
          if (lane == 0) fst[st0 + q * NW] = sm;
        }
      }
    }
    for (int st = st0; st < b1; st += NW) {
      float x[8];
      step_weights<TE, kF>(gp, gq, dp, dq, residual, st * kStep + lane * 8, V, x, off);
      float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
      sm = warp_sum(sm);
      if (lane == 0) fst[st] = sm;
    }
  } else {
    // a step of a filtered p row whose 512-entry block lies below the
    // threshold has no positive weight: its total is 0 without a load
    auto dead = [&](int st) { return bmp && to_f32(bmp[st >> 1]) < dp.thr; };
    if (!dp.onehot && (!residual || !dq.onehot)) {
      for (; st0 + (kU - 1) * NW < nfull; st0 += NW * kU) {
        Raw8<TE> rp[kU], rq[kU];
        bool dd[kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int base = (st0 + q * NW) * kStep + lane * 8;
          dd[q] = dead(st0 + q * NW);
          if (!dd[q]) {
            rp[q].load(gp + (base - off));
            if (residual) rq[q].load(gq + (base - off));
          }
        }
#pragma unroll
        for (int q = 0; q < kU; ++q) {
          const int base = (st0 + q * NW) * kStep + lane * 8;
          float sm = 0.f;
          if (!dd[q]) {
            float zp[8], zq[8], x[8];
            rp[q].get(zp);
            rq[q].get(zq);
            weights8<kF>(dp, dq, residual, base, zp, zq, x);
            sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
            sm = warp_sum(sm);
          }
          if (lane == 0) fst[st0 + q * NW] = sm;
        }
      }
    }
    for (int st = st0; st < b1; st += NW) {
      float sm = 0.f;
      if (!dead(st)) {
        float x[8];
        step_weights<TE, kF>(gp, gq, dp, dq, residual, st * kStep + lane * 8, V, x, off);
        sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
        sm = warp_sum(sm);
      }
      if (lane == 0) fst[st] = sm;
    }
  }
}

// Rows of a sequence's draw position j.
template <typename TE>
__device__ __forceinline__ void draw_rows(const Params &P, int s, int j, const TE *&gp,
                                          const TE *&gq) {
  gp = static_cast<const TE *>(
      row_ptr(P.target, static_cast<long long>(s) * (P.gamma + 1) + j, P.ld_t, sizeof(TE)));
  gq = static_cast<const TE *>(row_ptr(
      P.draft, static_cast<long long>(s) * P.gamma + (j < P.gamma ? j : 0), P.ld_d, sizeof(TE)));
}

// Double-float weights of the 8 entries from `base` (precise redraw).  Runs
// once per call site and step, so the entry loop stays rolled: unrolled, its
// code would come from the instruction cache's misses.
template <typename TE>
__device__ __forceinline__ void pweights8(const TE *gp, const TE *gq, const HpRow &rp,
                                          const HpRow &rq, int residual, Df rho, int base, int V,
                                          bool vec, const float *th, const float *tl,
                                          Df w[8]) {
  float zp[8], zq[8];
  hp_load8<TE>(gp, base, V, vec, zp);
  if (residual) hp_load8<TE>(gq, base, V, vec, zq);
#pragma unroll 1
  for (int e = 0; e < 8; ++e) {
    const Df ep = hp_exp(rp, zp[e], th, tl);
    if (!residual || ep.hi == 0.f) {
      w[e] = ep;
      continue;
    }
    const Df eq = hp_exp(rq, zq[e], th, tl);
    const Df d = df_sub(ep, df_mul(rho, eq));
    w[e] = d.hi > 0.f ? d : Df{0.f, 0.f};
  }
}

// ---------------------------------------------------------------------------
// 3. draw kernel: the search
// ---------------------------------------------------------------------------

// Shared state of a draw-kernel CTA (the step totals are dynamic shared
// memory: see chain_draw_kernel).
struct DrawShared {
  unsigned long long rr[kCMaxRows];  // merged row records
  PassSeq ps;                        // the draw's description
  DecideIn in[32];                   // the decision's inputs, one per lane of warp 0
  Df wsum[kDWarps];                  // search: per-warp sums of the step totals
  int wlast[kDWarps];                // search: per-warp last step with positive total
  int wfirst[kDWarps];               // search: per-warp first thread whose run crosses u W
  int step;
  float trel;
  int exact;
  double W;
  int token;
  float margin;
};

// Inverse-CDF search over the step totals tot[0, nsteps) (the whole CTA): a
// double-float prefix over the threads' runs of steps finds the step holding
// u * W, one warp scan of its weights the token.  The token goes to sh.token
// (-1: no positive weight), the total to sh.W and the distance of the draw
// from the nearer boundary of its token to sh.margin.
template <typename TE, bool kF>
__device__ void step_search(DrawShared &sh, const float *tot, int nsteps, const TE *gp,
                            const TE *gq, const RowDesc &dp, const RowDesc &dq, int residual,
                            int V, float u) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int per = (nsteps + kDThreads - 1) / kDThreads;
  const int s0 = min(nsteps, t * per), s1 = min(nsteps, s0 + per);
  Df seg{0.f, 0.f};
  int lastpos = -1;
  for (int st = s0; st < s1; ++st) {
    const float x = tot[st];
    seg = df_add(seg, Df{x, 0.f});
    if (x > 0.f) lastpos = st;
  }
  Df incl = seg;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const Df y = df_shfl_up(incl, off);
    if (lane >= off) incl = df_add(incl, y);
  }
  const int wl = warp_max_i(lastpos);
  if (lane == 31) sh.wsum[w] = incl;
  if (lane == 0) sh.wlast[w] = wl;
  wsync();
  // the warps' sums in a fixed order: every thread gets the same total
  Df base{0.f, 0.f}, W{0.f, 0.f};
  int last = -1;
#pragma unroll
  for (int x = 0; x < kDWarps; ++x) {
    if (x == w) base = W;
    W = df_add(W, sh.wsum[x]);
    last = max(last, sh.wlast[x]);
  }
  incl = df_add(base, incl);
  const Df tt = df_mul(Df{u, 0.f}, W);
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, df_gt(incl, tt) && seg.hi > 0.f);
  if (lane == 0) sh.wfirst[w] = hit ? __ffs(hit) - 1 : 32;
  wsync();
  int first = -1;
#pragma unroll
  for (int x = kDWarps - 1; x >= 0; --x)
    if (sh.wfirst[x] < 32) first = x * 32 + sh.wfirst[x];
  if (first < 0) {
    if (t == 0) {
      sh.step = last;
      sh.trel = 0.f;
      sh.exact = 0;
    }
  } else if (t == first) {
    Df acc = df_sub(incl, seg);
    int step = -1;
    float trel = 0.f;
    for (int st = s0; st < s1; ++st) {
      const float x = tot[st];
      const Df nx = df_add(acc, Df{x, 0.f});
      if (df_gt(nx, tt) && x > 0.f) {
        step = st;
        const Df r = df_sub(tt, acc);
        trel = r.hi + r.lo;
        break;
      }
      acc = nx;
    }
    sh.step = step < 0 ? lastpos : step;
    sh.trel = trel;
    sh.exact = step < 0 ? 0 : 1;
  }
  wsync();
  if (w == 0) {
    const int step = sh.step;
    const bool exact = sh.exact != 0;
    int token = -1;
    float margin = 0.f;
    if (step >= 0) {
      const float tr = sh.trel;
      const int base8 = step * kStep + lane * 8;
      float x[8];
      step_weights<TE, kF>(gp, gq, dp, dq, residual, base8, V, x);
      float sm = 0.f;
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sm += x[e];
        if (x[e] > 0.f) lp = base8 + e;
      }
      float fin = sm;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xFFFFFFFFu, fin, off);
        if (lane >= off) fin += y;
      }
      const float excl = fin - sm;
      const unsigned h2 = exact ? __ballot_sync(0xFFFFFFFFu, fin > tr && sm > 0.f) : 0u;
      if (h2) {
        const int f2 = __ffs(h2) - 1;
        int found = -1;
        float mg = 0.f;
        if (lane == f2) {
          float run = excl;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float prev = run;
            run += x[e];
            if (found < 0 && x[e] > 0.f && run > tr) {
              found = base8 + e;
              mg = fminf(tr - prev, run - tr);
            }
          }
          if (found < 0) found = lp;
        }
        token = __shfl_sync(0xFFFFFFFFu, found, f2);
        margin = __shfl_sync(0xFFFFFFFFu, mg, f2);
      } else {
        token = warp_max_i(lp);
        margin = 0.f;
      }
    }
    if (lane == 0) {
      sh.W = static_cast<double>(W.hi) + static_cast<double>(W.lo);
      sh.token = token;
      sh.margin = margin;
    }
  }
  wsync();
}

// One cluster of C CTAs per sequence (grid: nseq * C CTAs), every CTA of the
// cluster resident at once for the batches the path is built for.  Dynamic
// shared memory: the step totals tot[steps] (CTA 0 gathers all of them) and
// room for kDrawRecords row records.
template <typename TE, bool kFilt>
__global__ void __launch_bounds__(kDThreads, 7) chain_draw_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char draw_smem[];
  __shared__ DrawShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int seq = static_cast<int>(blockIdx.x) / C;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nsteps = P.steps;
  float *tot = reinterpret_cast<float *>(draw_smem);
  unsigned long long *srec = reinterpret_cast<unsigned long long *>(
      draw_smem + (static_cast<size_t>(nsteps) * sizeof(float) + 15) / 16 * 16);
  // every CTA of the cluster has started before the first remote access: the
  // arrive here pairs with the first wait below
  cluster_arrive();
  launch_dependents();
  // the decision's inputs (tokens, their logits, the uniforms) do not depend
  // on the rows kernel: CTA 0 loads them while it drains
  if (rank == 0 && warp == 0) sh.in[lane] = decide_inputs<TE>(P, seq);
  grid_dependency_wait();  // the rows kernel's records are visible
  // 1. the decision.  CTA r merges rows r, r + C, ... (records staged in
  // shared memory with all loads in flight at once when they fit) and puts
  // the merged records into CTA 0, which decides and hands the draw's
  // description to every CTA.
  const int rps = 2 * P.gamma + 1;
  const int R = P.cpr * kChainRecordsPerChunk;
  const int nmine = rank < rps ? (rps - 1 - rank) / C + 1 : 0;  // rows rank, rank + C, ...
  const int nrec = nmine * R;
  const bool staged = nrec <= kDrawRecords;
  if (staged) {
    for (int x0 = threadIdx.x; x0 < nrec; x0 += 4 * kDThreads) {
      unsigned long long b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = x0 + q * kDThreads;
        const int r = rank + (x / R) * C;
        b[q] = x < nrec ? __ldcg(P.srec + (static_cast<long long>(seq) * rps + r) * R + x % R)
                        : 0ull;
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (x0 + q * kDThreads < nrec) srec[x0 + q * kDThreads] = b[q];
    }
    __syncthreads();
  }
  unsigned long long *rr0 = cluster.map_shared_rank(sh.rr, 0);
  for (int k = warp; k < nmine; k += kDWarps) {
    const int r = rank + k * C;
    const unsigned long long *src =
        staged ? srec + static_cast<long long>(k) * R
               : P.srec + (static_cast<long long>(seq) * rps + r) * R;
    const unsigned long long rec = merge_row(P, seq, r, src, staged);
    if (lane == 0) sh.rr[r] = rec;  // staged locally, pushed after the first wait
  }
  __syncthreads();
  cluster_wait();  // every CTA has started
  if (rank != 0)
    for (int k = threadIdx.x; k < nmine; k += kDThreads) rr0[rank + k * C] = sh.rr[rank + k * C];
  cluster_sync_all();  // CTA 0 holds every merged record
  if (rank == 0) {
    if (warp == 0) decide_seq<TE, kFilt>(P, seq, sh.rr, sh.in[lane], true, sh.ps);
    __syncthreads();
    // the description to every other CTA (as 32-bit words)
    constexpr int kWords = static_cast<int>(sizeof(PassSeq) / 4);
    static_assert(sizeof(PassSeq) % 4 == 0, "PassSeq is copied as 32-bit words");
    for (int x = threadIdx.x; x < (C - 1) * kWords; x += kDThreads) {
      const int r = 1 + x / kWords, k = x % kWords;
      cluster.map_shared_rank(reinterpret_cast<uint32_t *>(&sh.ps), r)[k] =
          reinterpret_cast<const uint32_t *>(&sh.ps)[k];
    }
  }
  cluster_sync_all();  // every CTA holds the description
  PassSeq ps = sh.ps;
  if (!ps.draw) return;  // CTA 0 wrote the outputs (every CTA returns here)
  // 2. step totals of this CTA's steps, pushed into CTA 0's array
  const int per = (nsteps + C - 1) / C;
  const int b0 = min(nsteps, rank * per), b1 = min(nsteps, b0 + per);
  const TE *gp, *gq;
  draw_rows<TE>(P, seq, ps.j, gp, gq);
  const TE *bmp = kFilt ? static_cast<const TE *>(P.bmax) +
                              static_cast<long long>(seq * rps + ps.j) * P.nblk
                        : nullptr;  // block maxima of the p row (filtered calls)
  step_totals<TE, kDWarps, kFilt>(gp, gq, ps.dp, ps.dq, ps.residual, P.V, b0, b1, tot, bmp);
  __syncthreads();
  if (rank != 0) {
    float *dst = cluster.map_shared_rank(tot, 0);
    for (int st = b0 + threadIdx.x; st < b1; st += kDThreads) dst[st] = tot[st];
    cluster_arrive();  // release: CTA 0 reads the totals after its wait
    return;
  }
  cluster_arrive();
  cluster_wait();
  // 3. the search (CTA 0)
  step_search<TE, kFilt>(sh, tot, nsteps, gp, gq, ps.dp, ps.dq, ps.residual, P.V, ps.u);
  int token = sh.token;
  double W = sh.W;
  float margin = sh.margin;
  if (ps.residual && !(W > 0.0)) {
    // degenerate residual: draw from p itself (this CTA sums the whole row)
    ps.flags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
    ps.residual = 0;
    ps.dq = ps.dp;
    ps.dq.onehot = 1;
    ps.dq.a = 0;
    step_totals<TE, kDWarps, kFilt>(gp, gq, ps.dp, ps.dq, 0, P.V, 0, nsteps, tot, bmp);
    __syncthreads();
    step_search<TE, kFilt>(sh, tot, nsteps, gp, gq, ps.dp, ps.dq, 0, P.V, ps.u);
    token = sh.token;
    W = sh.W;
    margin = sh.margin;
  }
  if (token < 0) token = ps.dp.a;  // no positive weight at all (not reachable with finite rows)
  // a draw within 1e-6 of the draw mass of a boundary is queued for the
  // precise kernel (the single-precision boundary error measured on
  // 128K-entry rows stays below 3e-7 of it)
  const int near = margin < 1e-6f * static_cast<float>(W) ? 1 : 0;
  if (threadIdx.x == 0) {
    ps.W = static_cast<float>(W);
    write_outputs(P, seq, ps, token, W, near);
    if (near) {
      reinterpret_cast<PassSeq *>(P.pseqw)[seq] = ps;
      const uint32_t q = atomicAdd(P.pctr, 1u);  // the queue is read after this kernel
      if (q < static_cast<uint32_t>(P.nseq)) P.near_list[q] = seq + 1;
    }
  }
}

// ---------------------------------------------------------------------------
// 4. precise kernel: one cluster per queued draw
// ---------------------------------------------------------------------------

struct PreciseShared {
  Df part[kPreciseCluster][2];  // every CTA's shares of S_p, S_q
  Df pred[2][kPWarps];
  Df wsum[kPWarps];             // search: per-warp sums
  int wfirst[kPWarps];          // search: per-warp first thread past the target
  int wlast[kPWarps];           // search: per-warp last positive index
  int step, exact;
  Df trel;
  float tab_hi[64], tab_lo[64];
};

// Inclusive double-float prefix of v over the CTA's threads (kPThreads), and
// the CTA total in `tot` (the same value in every thread: the warps' sums are
// added in a fixed order).
__device__ __forceinline__ Df block_df_scan(PreciseShared &sh, Df v, Df &tot) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  Df incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const Df y = df_shfl_up(incl, off);
    if (lane >= off) incl = df_add(incl, y);
  }
  if (lane == 31) sh.wsum[w] = incl;
  __syncthreads();
  Df base{0.f, 0.f}, T{0.f, 0.f};
  for (int x = 0; x < kPWarps; ++x) {
    if (x == w) base = T;
    T = df_add(T, sh.wsum[x]);
  }
  tot = T;
  return df_add(base, incl);
}

// The first thread of the CTA for which `hit` holds (-1: none), and the
// largest `idx` of the CTA (-1 when every idx is -1).
__device__ __forceinline__ int block_first(PreciseShared &sh, bool hit, int idx, int &last) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
  const int wl = warp_max_i(idx);
  if (lane == 0) {
    sh.wfirst[w] = b ? __ffs(b) - 1 : 32;
    sh.wlast[w] = wl;
  }
  __syncthreads();
  int first = -1;
  last = -1;
  for (int x = kPWarps - 1; x >= 0; --x) {
    if (sh.wfirst[x] < 32) first = x * 32 + sh.wfirst[x];
    last = max(last, sh.wlast[x]);
  }
  __syncthreads();  // sh.wfirst / wlast are reused by the next call
  return first;
}

// Per 256-entry step of this CTA's steps [b0, b1): the double-float sums A of
// e_p and B of e_q over the entries whose weight e_p - rho e_q is certainly
// positive, classified with the single-precision rho of the row statistics
// (within 1e-6 of the exact one; an entry is certain when
// |e_p - rho e_q| > 1e-5 e_p), or B = -1 when an entry of the step is
// uncertain; and the CTA's shares of S_p and S_q into sh.pred.  A draw from p
// stores A = the sum of e_p, B = 0.  The step loop stays rolled (its body is
// long: unrolled, the code would miss the instruction cache once per step)
// and loads the warp's next step while it computes this one.
template <typename TE>
__device__ void precise_steps(PreciseShared &sh, const PassSeq &ps, const TE *gp, const TE *gq,
                              const HpRow &rp, const HpRow &rq, bool vec, int V, int b0, int b1,
                              float2 *sa, float2 *sb) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int residual = ps.residual;
  const float rho_a = residual ? ps.dq.invS / ps.dp.invS : 0.f;  // S_p / S_q, single precision
  Df sp_tot{0.f, 0.f}, sq_tot{0.f, 0.f};
  float np[8], nq[8];
  int st = b0 + w;
  if (st < b1) {
    hp_load8<TE>(gp, st * kStep + lane * 8, V, vec, np);
    if (residual) hp_load8<TE>(gq, st * kStep + lane * 8, V, vec, nq);
  }
#pragma unroll 1
  for (; st < b1; st += kPWarps) {
    float zp[8], zq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      zp[e] = np[e];
      zq[e] = residual ? nq[e] : 0.f;
    }
    const int nx = st + kPWarps;
    if (nx < b1) {
      hp_load8<TE>(gp, nx * kStep + lane * 8, V, vec, np);
      if (residual) hp_load8<TE>(gq, nx * kStep + lane * 8, V, vec, nq);
    }
    Df ep[8], eq[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      ep[e] = hp_exp(rp, zp[e], sh.tab_hi, sh.tab_lo);
      eq[e] = residual ? hp_exp(rq, zq[e], sh.tab_hi, sh.tab_lo) : Df{0.f, 0.f};
    }
    Df sp{0.f, 0.f}, sq{0.f, 0.f}, a{0.f, 0.f}, b{0.f, 0.f};
    bool unc = false;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      sp = df_add(sp, ep[e]);
      if (!residual) continue;
      sq = df_add(sq, eq[e]);
      if (ep[e].hi > 0.f) {
        const float d = fmaf(-rho_a, eq[e].hi, ep[e].hi);
        if (d > 1e-5f * ep[e].hi) {
          a = df_add(a, ep[e]);
          b = df_add(b, eq[e]);
        } else if (d >= -1e-5f * ep[e].hi) {
          unc = true;
        }
      }
    }
    const Df A = df_warp_sum(residual ? a : sp);
    const Df Bq = df_warp_sum(b);
    unc = __any_sync(0xFFFFFFFFu, unc);
    if (lane == 0) {
      sa[st] = make_float2(A.hi, A.lo);
      sb[st] = unc ? make_float2(-1.f, 0.f) : make_float2(Bq.hi, Bq.lo);
    }
    sp_tot = df_add(sp_tot, sp);
    sq_tot = df_add(sq_tot, sq);
  }
  sp_tot = df_warp_sum(sp_tot);
  sq_tot = df_warp_sum(sq_tot);
  if (lane == 0) {
    sh.pred[0][w] = sp_tot;
    sh.pred[1][w] = sq_tot;
  }
  __syncthreads();
}

// CTA 0 (every thread), after every CTA's step sums are in sa / sb: a
// double-float prefix of A - rho B over the threads' runs of steps finds the
// step holding u Z, then a double-float prefix of the step's 256 weights (one
// entry a thread) the token (-1: no positive weight).  All sums are
// double-float (about 48 significant bits).
template <typename TE>
__device__ int precise_search(PreciseShared &sh, const float2 *sa, const float2 *sb, int nsteps,
                              const PassSeq &ps, Df rho, const TE *gp, const TE *gq,
                              const HpRow &rp, const HpRow &rq, int V) {
  const int t = threadIdx.x;
  const int per = (nsteps + kPThreads - 1) / kPThreads;
  const int s0 = min(nsteps, t * per), s1 = min(nsteps, s0 + per);
  const Df nrho{-rho.hi, -rho.lo};
  Df seg{0.f, 0.f};
  int lastpos = -1;
  for (int st = s0; st < s1; ++st) {
    const Df x = df_add(Df{sa[st].x, sa[st].y}, df_mul(nrho, Df{sb[st].x, sb[st].y}));
    seg = df_add(seg, x);
    if (x.hi > 0.f) lastpos = st;
  }
  Df Z;
  const Df incl = block_df_scan(sh, seg, Z);
  const Df tt = df_mul(Df{ps.u, 0.f}, Z);
  int last;
  const int first = block_first(sh, df_gt(incl, tt) && seg.hi > 0.f, lastpos, last);
  if (first < 0) {
    if (t == 0) {
      sh.step = last;
      sh.exact = 0;
    }
  } else if (t == first) {
    Df acc = df_sub(incl, seg);
    int step = -1;
    for (int st = s0; st < s1 && step < 0; ++st) {
      const Df x = df_add(Df{sa[st].x, sa[st].y}, df_mul(nrho, Df{sb[st].x, sb[st].y}));
      if (df_gt(df_add(acc, x), tt) && x.hi > 0.f) {
        step = st;
        sh.trel = df_sub(tt, acc);
      }
      acc = df_add(acc, x);
    }
    sh.step = step < 0 ? lastpos : step;
    sh.exact = step < 0 ? 0 : 1;
  }
  __syncthreads();
  const int step = sh.step;
  if (step < 0) return -1;
  const bool exact = sh.exact != 0;
  const Df trel = sh.trel;
  // the step's weights, one entry a thread
  const int v = step * kStep + t;
  Df wv{0.f, 0.f};
  if (t < kStep && v < V) {
    const Df ep = hp_exp(rp, to_f32(gp[v]), sh.tab_hi, sh.tab_lo);
    if (!ps.residual || ep.hi == 0.f) {
      wv = ep;
    } else {
      const Df eq = hp_exp(rq, to_f32(gq[v]), sh.tab_hi, sh.tab_lo);
      const Df d = df_sub(ep, df_mul(rho, eq));
      wv = d.hi > 0.f ? d : Df{0.f, 0.f};
    }
  }
  Df Ts;
  const Df cum = block_df_scan(sh, wv, Ts);
  const bool pos = wv.hi > 0.f;
  int lp;
  const int f = block_first(sh, exact && pos && df_gt(cum, trel), pos ? v : -1, lp);
  return f >= 0 ? step * kStep + f : lp;
}

// Clusters of Cp CTAs (grid: kPreciseGrid * Cp CTAs); cluster y redraws the
// queued draws y, y + kPreciseGrid, ... : double-float step sums of each
// CTA's steps; the exact rho = S_p / S_q from every CTA's shares; exact totals
// of the steps an entry of which was uncertain; then CTA 0 searches and
// overwrites the token.  Dynamic shared memory: sa[steps], sb[steps].
template <typename TE>
__global__ void __launch_bounds__(kPThreads, 2) chain_precise_kernel(const Params P,
                                                                     const Exp2Table tab) {
  extern __shared__ __align__(16) unsigned char precise_smem[];
  __shared__ PreciseShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int y = static_cast<int>(blockIdx.x) / C, ny = static_cast<int>(gridDim.x) / C;
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int V = P.V, nsteps = P.steps;
  float2 *sa = reinterpret_cast<float2 *>(precise_smem);
  float2 *sb = sa + nsteps;
  cluster_arrive();
  launch_dependents();
  if (t < 64) {
    sh.tab_hi[t] = tab.hi[t];
    sh.tab_lo[t] = tab.lo[t];
  }
  grid_dependency_wait();  // the draw kernel's queue is complete
  const int count = static_cast<int>(min(__ldcg(P.pctr), static_cast<uint32_t>(P.nseq)));
  if (y >= count) return;  // every CTA of this cluster returns
  cluster_wait();
  __syncthreads();
  const int per = (nsteps + C - 1) / C;
  const int b0 = min(nsteps, rank * per), b1 = min(nsteps, b0 + per);
  for (int item = y; item < count; item += ny) {
    const int s = __ldcg(P.near_list + item) - 1;  // written by the draw kernel
    const bool ok = s >= 0 && s < P.nseq;
    const PassSeq ps = ok ? reinterpret_cast<const PassSeq *>(P.pseqw)[s] : PassSeq{};
    // an entry outside the batch or a position that is not a draw is skipped
    // (the same decision in every CTA, so the barriers below still pair up)
    const bool run = ok && ps.j >= 0 && ps.j <= P.gamma;
    const TE *gp = nullptr, *gq = nullptr;
    if (run) draw_rows<TE>(P, s, ps.j, gp, gq);
    const bool vec =
        ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(gq)) & 15u) == 0;
    const HpRow rp = hp_row(ps.dp, run ? __ldg(P.Tp + s) : 1.f);
    const HpRow rq = ps.residual ? hp_row(ps.dq, run ? __ldg(P.Tq + s) : 1.f) : rp;
    if (run) {
      precise_steps<TE>(sh, ps, gp, gq, rp, rq, vec, V, b0, b1, sa, sb);
      // this CTA's shares to every CTA; its step sums to CTA 0
      if (t < C) {
        Df A{0.f, 0.f}, B{0.f, 0.f};
        for (int x = 0; x < kPWarps; ++x) {
          A = df_add(A, sh.pred[0][x]);
          B = df_add(B, sh.pred[1][x]);
        }
        Df *dst = cluster.map_shared_rank(&sh.part[0][0], t);
        dst[2 * rank] = A;
        dst[2 * rank + 1] = B;
      }
      if (rank != 0) {
        float2 *ra = cluster.map_shared_rank(sa, 0), *rb = cluster.map_shared_rank(sb, 0);
        for (int st = b0 + t; st < b1; st += kPThreads) {
          ra[st] = sa[st];
          rb[st] = sb[st];
        }
      }
    }
    cluster_sync_all();
    Df rho{0.f, 0.f};
    if (run && ps.residual) {
      // the exact normaliser ratio, summed in the same order in every CTA
      Df Sp{0.f, 0.f}, Sq{0.f, 0.f};
      for (int r = 0; r < C; ++r) {
        Sp = df_add(Sp, sh.part[r][0]);
        Sq = df_add(Sq, sh.part[r][1]);
      }
      // rho = Sp / Sq as a double-float: q1 = Sp.hi / Sq.hi, then one
      // correction step q2 = (Sp - q1 Sq) / Sq.hi
      const float q1 = __fdiv_rn(Sp.hi, Sq.hi);
      const Df r = df_sub(Sp, df_mul(Df{q1, 0.f}, Sq));
      const float q2 = __fdiv_rn(r.hi, Sq.hi);
      rho = df_norm(q1, q2);
      // uncertain steps of this CTA (B < 0): their exact totals, one warp per step
      float2 *ra = cluster.map_shared_rank(sa, 0), *rb = cluster.map_shared_rank(sb, 0);
      for (int base = b0 + w * 32; base < b1; base += kPWarps * 32) {
        const int st = base + lane;
        unsigned todo = __ballot_sync(0xFFFFFFFFu, st < b1 && sb[st].x < 0.f);
        while (todo) {
          const int x = base + __ffs(todo) - 1;
          todo &= todo - 1;
          Df wd[8];
          pweights8<TE>(gp, gq, rp, rq, 1, rho, x * kStep + lane * 8, V, vec, sh.tab_hi,
                        sh.tab_lo, wd);
          Df acc{0.f, 0.f};
#pragma unroll
          for (int e = 0; e < 8; ++e) acc = df_add(acc, wd[e]);
          acc = df_warp_sum(acc);
          if (lane == 0) {
            ra[x] = make_float2(acc.hi, acc.lo);
            rb[x] = make_float2(0.f, 0.f);
          }
        }
      }
    }
    cluster_sync_all();
    if (run && rank == 0) {
      const int token = precise_search<TE>(sh, sa, sb, nsteps, ps, rho, gp, gq, rp, rq, V);
      if (t == 0 && token >= 0) {
        const long long obase = static_cast<long long>(s) * (P.gamma + 1);
        P.out_tokens[obase + ps.j] = token;
        P.outs[obase + ps.j].token = token;
      }
    }
    cluster_sync_all();  // CTA 0 has read sa / sb before the next item writes them
  }
}

// ---------------------------------------------------------------------------
// 5. tree walk kernel: one cluster per tree
// ---------------------------------------------------------------------------

constexpr int kWWarps = 8;
constexpr int kWThreads = kWWarps * 32;
constexpr int kWalkCluster = 8;  // CTAs per tree (fewer when such a cluster cannot run)
static_assert(kWalkMaxNodes <= 2 * kWThreads, "the shape pass takes two nodes a thread");
static_assert(kWThreads >= kDThreads, "the draw search runs on the first kDThreads threads");

struct WalkShared {
  unsigned long long rr[2 * kWalkMaxNodes];  // merged records: target rows, then draft rows
  int par[kWalkMaxNodes];                    // parent of each node
  int kids[kWalkMaxNodes];                   // children of the current node, ascending
  int path[kWalkMaxNodes];                   // the walked path, root first
  int rows[2 * kWalkMaxNodes];               // the rows that have records
  int cx[kWalkMaxNodes];                     // per node c: its token x, the logits of x in
  float czp[kWalkMaxNodes], czq[kWalkMaxNodes];  //   its parent's target and draft rows,
  float cua[kWalkMaxNodes], cud[kWalkMaxNodes];  //   its acceptance and draw uniforms
  Df part[2][kMaxCluster];                   // every CTA's share of a pass total (by parity)
  RowDesc dp, dq;                            // the current node's rows
  int nk, nrows, accept;
  uint32_t tf;
};

__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)),
               "l"(__cvta_generic_to_global(src))
               : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// This CTA's share of the steps of a row of V entries split over C CTAs:
// steps [b0, b1), and whether both rows' shares fit in the staging buffer.
struct WalkShare {
  int b0, b1, cap;  // cap: entries of a row the buffer holds
  bool staged;
};
template <typename TE>
__device__ __forceinline__ WalkShare walk_share(int C, int rank, int nsteps, int bufcap) {
  WalkShare w;
  const int per = (nsteps + C - 1) / C;
  w.b0 = min(nsteps, rank * per);
  w.b1 = min(nsteps, w.b0 + per);
  w.cap = per * kStep;
  w.staged = w.cap * static_cast<int>(sizeof(TE)) * 2 <= bufcap;
  return w;
}

// Start copying this CTA's share of a node's target row (and of its draft row
// when `withq`) into the staging buffer: 16-byte asynchronous copies, all in
// flight at once (every thread); walk_pass waits for them.  The ragged tail
// of the row (less than 16 bytes) is copied with plain loads.
template <typename TE>
__device__ void walk_prefetch(const WalkShare &sh, TE *buf, const TE *gp, const TE *gq, bool withq,
                              int V) {
  constexpr int kPer16 = 16 / static_cast<int>(sizeof(TE));
  TE *sp = buf, *sq = buf + sh.cap;
  const int e0 = sh.b0 * kStep;
  const int n = max(0, min(V, sh.b1 * kStep) - e0);
  const int nvec = n / kPer16;
  for (int i = threadIdx.x; i < nvec; i += kWThreads) {
    cp_async16(sp + i * kPer16, gp + e0 + i * kPer16);
    if (withq) cp_async16(sq + i * kPer16, gq + e0 + i * kPer16);
  }
  for (int v = nvec * kPer16 + threadIdx.x; v < n; v += kWThreads) {
    sp[v] = gp[e0 + v];
    if (withq) sq[v] = gq[e0 + v];
  }
}

// One pass of the cluster over the current node's rows (every thread of every
// CTA): the 256-entry step totals of the draw weights [p - c q]_+ (p itself
// for c = 0) of this CTA's share of the steps, into CTA 0's array, and the
// total over the row, the same double-float in every CTA (each CTA's share,
// lane 0's value, added in rank order).  A staged share is read from the
// staging buffer, which walk_prefetch filled before the first pass at the
// node (every later pass at the node reads the same copy); else from global
// memory.
// `parity` alternates between consecutive passes: a CTA reads the shares of a
// pass before it arrives at the next pass's barrier, so the pass after next
// may overwrite them.
template <typename TE>
__device__ Df walk_pass(WalkShared &ws, cg::cluster_group &cluster, const WalkShare &sr, int C,
                        int rank, float *tot, const TE *buf, const TE *gp, const TE *gq,
                        const RowDesc &dp, const RowDesc &dq, float c, int V, int parity) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int b0 = sr.b0, b1 = sr.b1;
  const int residual = c > 0.f ? 1 : 0;
  RowDesc dqc = dq;
  if (residual && !dq.onehot) dqc.invS = dq.invS * c;  // c q_v = 2^((z - m) k) (c / S_q)
  if (sr.staged) {
    cp_async_wait_all();
    __syncthreads();
    step_totals<TE, kWWarps, false>(buf, buf + sr.cap, dp, dqc, residual, V, b0, b1, tot,
                                    nullptr, b0 * kStep);
  } else {
    step_totals<TE, kWWarps, false>(gp, gq, dp, dqc, residual, V, b0, b1, tot);
  }
  __syncthreads();
  if (warp == 0) {
    Df s{0.f, 0.f};
    for (int st = b0 + lane; st < b1; st += 32) s = df_add(s, Df{tot[st], 0.f});
    s = df_shfl(df_warp_sum(s), 0);  // lane 0's value, sent to every CTA
    if (lane < C) cluster.map_shared_rank(&ws.part[parity][0], lane)[rank] = s;
  }
  if (rank != 0) {
    float *dst = cluster.map_shared_rank(tot, 0);
    for (int st = b0 + tid; st < b1; st += kWThreads) dst[st] = tot[st];
  }
  cluster_sync_all();
  Df W{0.f, 0.f};
  for (int r = 0; r < C; ++r) W = df_add(W, ws.part[parity][r]);
  return W;
}

// Outputs of a walked tree (every thread of CTA 0): the path, the accepted
// tokens and the final token at position `depth`, and the final unit's record
// that the refine and residual-output kernels read.
__device__ void walk_outputs(const Params &P, const WalkShared &ws, int tree, int depth,
                             int token, uint32_t flags, const RowDesc &dp, const RowDesc &dq,
                             float c, float total, int kind, int nres, int near) {
  const int N = P.ups;
  const long long nbase = static_cast<long long>(tree) * N;
  const int width = P.max_depth + 1;
  const long long obase = static_cast<long long>(tree) * width;
  for (int i = threadIdx.x; i < width; i += kWThreads) {
    P.out_path[obase + i] = i <= depth ? ws.path[i] : -1;
    int v = -1;
    if (i < depth) v = ws.cx[ws.path[i + 1]];
    else if (i == depth) v = token;
    P.out_tokens[obase + i] = v;
  }
  if (threadIdx.x == 0) {
    const int cur = ws.path[depth];
    const long long unit = nbase + cur;
    P.out_num[tree] = depth;
    if (P.out_flags) P.out_flags[tree] = flags;
    UnitOut o;
    o.next = -1;
    o.token = token;
    o.flags = flags;
    o.near = near;
    P.outs[unit] = o;
    UnitStats st;
    st.p = dp;
    st.q = dq;
    st.c = c;
    st.total = total;
    st.kind = kind;
    st.node = cur;
    st.n_res = nres;
    st.pad = 0;
    P.stats[unit] = st;
    P.final_unit[tree] = static_cast<int>(unit);
    queue_refine(P, tree, unit, depth, near);
  }
}

// A tree without a walk (every thread of CTA 0): an invalid tree (num = -1)
// or a bounded wait of the rows kernel that gave up (num = 0); every path
// entry and token -1.
__device__ void walk_no_result(const Params &P, int tree, int num, uint32_t flags) {
  const int width = P.max_depth + 1;
  const long long obase = static_cast<long long>(tree) * width;
  for (int i = threadIdx.x; i < width; i += kWThreads) {
    P.out_path[obase + i] = -1;
    P.out_tokens[obase + i] = -1;
  }
  if (threadIdx.x == 0) {
    P.out_num[tree] = num;
    if (P.out_flags) P.out_flags[tree] = flags;
    P.final_unit[tree] = -1;
  }
}

// One cluster of C CTAs per tree (grid: T * C CTAs), after the rows kernel
// has left the records of the tree's N target rows and of the draft rows of
// its internal nodes.  Every CTA merges its share of the rows and hands the
// merged records to every CTA; then all CTAs walk the tree together, taking
// the same decisions from the same data: at node n with sampled p, child
// tokens are tested in ascending id against the held distribution
// [p - c q]_+ / M (p itself before the first rejection: c = 0, M = 1), each
// rejection followed by one pass of the cluster over n's rows for the next
// multiplier c' = c + M and its total M' (a zero M' keeps the held
// distribution and flags the residual degenerate); a greedy p accepts the
// first child equal to its argmax.  Only the nodes on the walked path are
// ever touched.  The final draw (every child rejected, or a leaf's bonus
// draw from p) is CTA 0's double-float search over the step totals of the
// last pass; a draw within the refine guard of a boundary is queued for the
// refine kernel, which recomputes the multipliers in double precision.
// Dynamic shared memory: the step totals tot[steps], then a staging buffer of
// P.walk_buf bytes (the records while they are merged, then each pass's share
// of the rows).
template <typename TE>
__global__ void __launch_bounds__(kWThreads, 2) tree_walk_kernel(const Params P) {
  extern __shared__ __align__(16) unsigned char walk_smem[];
  __shared__ WalkShared ws;
  __shared__ DrawShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int rank = static_cast<int>(cluster.block_rank());
  const int tree = static_cast<int>(blockIdx.x) / C;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.ups, V = P.V, nsteps = P.steps;
  const long long nbase = static_cast<long long>(tree) * N;
  float *tot = reinterpret_cast<float *>(walk_smem);
  unsigned char *bufb = walk_smem + (static_cast<size_t>(nsteps) * sizeof(float) + 15) / 16 * 16;
  unsigned long long *srec = reinterpret_cast<unsigned long long *>(bufb);
  TE *buf = reinterpret_cast<TE *>(bufb);
  // every CTA of the cluster has started before the first remote access: the
  // arrive here pairs with the first wait below
  cluster_arrive();
  launch_dependents();
  // 1. from the inputs alone: every node's acceptance-test inputs (all loads
  // in flight at once), and the tree's shape: every parent id below its
  // child's, every depth within max_depth (depths by pointer jumping, with
  // kids and path as scratch)
  int *anc = ws.kids, *dep = ws.path;
  int bad = 0;
  for (int n = tid; n < N; n += kWThreads) {
    const int a = __ldg(P.parent + nbase + n);
    const int x = __ldg(P.tokens + nbase + n);
    ws.par[n] = a;
    const bool link = n == 0 ? a == -1 : (a >= 0 && a < n);
    if (!link) bad = 1;
    anc[n] = n == 0 ? 0 : a;
    dep[n] = n == 0 ? 0 : 1;
    float zp = 0.f, zq = 0.f;
    if (n > 0 && link && x >= 0 && x < V) {
      zp = to_f32(static_cast<const TE *>(row_ptr(P.target, nbase + a, P.ld_t, sizeof(TE)))[x]);
      zq = to_f32(static_cast<const TE *>(row_ptr(P.draft, nbase + a, P.ld_d, sizeof(TE)))[x]);
    }
    ws.cx[n] = x;
    ws.czp[n] = zp;
    ws.czq[n] = zq;
    ws.cua[n] = unit_uniform(P, tree, n, 0);
    ws.cud[n] = unit_uniform(P, tree, n, 1);
  }
  uint32_t tflags = __syncthreads_or(bad) ? SPEC_FLAG_BAD_TREE : 0u;
  if (!tflags) {
    for (int span = 1; span < N; span <<= 1) {
      int la[2] = {0, 0}, ld[2] = {0, 0};
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int n = tid + i * kWThreads;
        if (n < N) {
          const int a = anc[n];
          la[i] = anc[a];
          ld[i] = dep[n] + dep[a];
        }
      }
      __syncthreads();
#pragma unroll
      for (int i = 0; i < 2; ++i) {
        const int n = tid + i * kWThreads;
        if (n < N) {
          anc[n] = la[i];
          dep[n] = ld[i];
        }
      }
      __syncthreads();
    }
    int deep = 0;
    for (int n = tid; n < N; n += kWThreads)
      if (dep[n] > P.max_depth) deep = 1;
    if (__syncthreads_or(deep)) tflags = SPEC_FLAG_DEPTH;
  }
  const float Tp = __ldg(P.Tp + tree), Tq = __ldg(P.Tq + tree);
  const bool p_arg = row_is_arg(Tp), q_arg = row_is_arg(Tq);
  const bool tp_bad = !(Tp >= 0.f) || Tp == INFINITY, tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  const float kp = p_arg ? 0.f : kLog2e / Tp, kq = q_arg ? 0.f : kLog2e / Tq;
  if (!tflags) {
    // the rows that have records: the N target rows, then the draft rows of
    // the nodes with children (none for a greedy target)
    for (int n = tid; n < N; n += kWThreads) dep[n] = 0;
    __syncthreads();
    for (int n = tid + 1; n < N; n += kWThreads) dep[ws.par[n]] = 1;
    __syncthreads();
    if (warp == 0) {
      int cnt = N;
      for (int base = 0; base < N; base += 32) {
        const int n = base + lane;
        if (n < N) ws.rows[n] = n;
        const bool has = n < N && !p_arg && dep[n] != 0;
        const unsigned b = __ballot_sync(0xFFFFFFFFu, has);
        if (has) ws.rows[cnt + __popc(b & ((1u << lane) - 1u))] = N + n;
        cnt += __popc(b);
      }
      if (lane == 0) ws.nrows = cnt;
    }
  }
  grid_dependency_wait();  // the rows kernel's records are visible
  if (tflags) {
    if (rank == 0) walk_no_result(P, tree, -1, tflags);
    return;  // every CTA of the cluster returns here
  }
  __syncthreads();
  // 2. CTA r merges listed rows r, r + C, ... (records staged in shared memory
  // with all loads in flight at once when they fit) and hands the merged
  // records to every CTA
  const int nrows = ws.nrows;
  const int rps = 2 * N;
  const int R = P.cpr * kChainRecordsPerChunk;
  const int nmine = rank < nrows ? (nrows - 1 - rank) / C + 1 : 0;
  const int nrec = nmine * R;
  const bool staged = static_cast<long long>(nrec) * 8 <= P.walk_buf;
  if (staged) {
    for (int x0 = tid; x0 < nrec; x0 += 4 * kWThreads) {
      unsigned long long b[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int x = x0 + q * kWThreads;
        b[q] = 0ull;
        if (x < nrec) {
          const int r = ws.rows[rank + (x / R) * C];
          b[q] = __ldcg(P.srec + (static_cast<long long>(tree) * rps + r) * R + x % R);
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (x0 + q * kWThreads < nrec) srec[x0 + q * kWThreads] = b[q];
    }
    __syncthreads();
  }
  for (int k = warp; k < nmine; k += kWWarps) {
    const int r = ws.rows[rank + k * C];
    const unsigned long long *src = staged ? srec + static_cast<long long>(k) * R
                                           : P.srec + (static_cast<long long>(tree) * rps + r) * R;
    const unsigned long long rec = merge_row(P, tree, r, src, staged);
    if (lane == 0) ws.rr[r] = rec;
  }
  __syncthreads();
  cluster_wait();  // every CTA has started
  for (int x = tid; x < nmine * C; x += kWThreads) {
    const int k = x / C, dst = x - k * C;
    if (dst == rank) continue;
    const int r = ws.rows[rank + k * C];
    cluster.map_shared_rank(ws.rr, dst)[r] = ws.rr[r];
  }
  cluster_sync_all();  // every CTA holds every merged record
  if (__ldcg(P.err)) {
    // a bounded wait of the rows kernel gave up: the documented fallback
    if (rank == 0) walk_no_result(P, tree, 0, SPEC_FLAG_TIMEOUT);
    return;
  }
  // 3. the walk
  if (tid == 0) ws.path[0] = 0;
  const WalkShare sr = walk_share<TE>(C, rank, nsteps, P.walk_buf);
  int cur = 0, depth = 0, parity = 0;
  int loaded = -1;  // the node whose rows the staging buffer holds
  uint32_t flags = 0u;
  for (;;) {
    const TE *gp = static_cast<const TE *>(row_ptr(P.target, nbase + cur, P.ld_t, sizeof(TE)));
    const TE *gq = static_cast<const TE *>(row_ptr(P.draft, nbase + cur, P.ld_d, sizeof(TE)));
    // the node's row descriptors and its children (warp 0)
    if (warp == 0) {
      RowDesc dp = row_desc(ws.rr[cur], p_arg, tp_bad, kp, V);
      if (!p_arg && dp.onehot) dp.a = warp_finite_argmax<TE>(gp, V);  // statistics not finite
      int nk = 0;
      for (int base = cur + 1; base < N; base += 32) {
        const int c = base + lane;
        const bool hit = c < N && ws.par[c] == cur;
        const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
        if (hit) ws.kids[nk + __popc(b & ((1u << lane) - 1u))] = c;
        nk += __popc(b);
      }
      RowDesc dq = dp;  // a one-hot stand-in where q is never read
      dq.onehot = 1;
      dq.a = 0;
      dq.flags = 0u;
      if (nk > 0 && !dp.onehot) {
        dq = row_desc(ws.rr[N + cur], q_arg, tq_bad, kq, V);
        if (!q_arg && dq.onehot) dq.a = warp_finite_argmax<TE>(gq, V);
      }
      if (lane == 0) {
        ws.dp = dp;
        ws.dq = dq;
        ws.nk = nk;
      }
    }
    __syncthreads();
    const RowDesc dp = ws.dp, dq = ws.dq;
    const int nk = ws.nk;
    flags |= dp.flags;
    int next = -1;
    if (dp.onehot) {
      // greedy rule: the first child whose token is p's argmax; q is not used
      for (int i = 0; i < nk; ++i) {
        const int x = ws.cx[ws.kids[i]];
        if (!(x >= 0 && x < V)) flags |= SPEC_FLAG_BAD_TOKEN;
        if (x == dp.a) {
          next = ws.kids[i];
          break;
        }
      }
      if (next < 0) {
        if (rank == 0) walk_outputs(P, ws, tree, depth, dp.a, flags, dp, dq, 0.f, 0.f,
                                    nk > 0 ? 1 : 0, 0, 0);
        return;
      }
    } else {
      float c = 0.f, M = 1.f;  // the held distribution [p - c q]_+ / M
      int nres = 0;
      bool held = false;  // CTA 0 holds the step totals of the held distribution
      if (nk > 0) flags |= dq.flags;
      for (int i = 0; i < nk; ++i) {
        if (tid == 0) {
          const int ch = ws.kids[i];
          const int x = ws.cx[ch];
          const float zp = ws.czp[ch], zq = dq.onehot ? 0.f : ws.czq[ch], ua = ws.cua[ch];
          uint32_t f = 0u;
          int acc = 0;
          if (!(x >= 0 && x < V)) {
            f = SPEC_FLAG_BAD_TOKEN;
          } else {
            const float px = pprob<false>(dp, zp, x);
            const float qx = pprob<false>(dq, zq, x);
            if (!(qx > 0.f)) {
              f = SPEC_FLAG_ZERO_Q;
            } else {
              const float w = c > 0.f ? fmaxf(fmaf(-c, qx, px), 0.f) / M : px;
              acc = ua < fminf(1.f, w / qx) ? 1 : 0;
            }
          }
          ws.accept = acc;
          ws.tf = f;
        }
        __syncthreads();
        flags |= ws.tf;
        if (ws.accept) {
          next = ws.kids[i];
          break;
        }
        // rejected: the residual for the next multiplier and its total (the
        // pass's barriers also order this read of ws.accept before the next
        // write)
        const float cn = c + M;
        if (sr.staged && loaded != cur) {  // the node's first pass: its rows to the buffer
          walk_prefetch<TE>(sr, buf, gp, gq, !dq.onehot, V);
          loaded = cur;
        }
        const Df W = walk_pass<TE>(ws, cluster, sr, C, rank, tot, buf, gp, gq, dp, dq, cn, V,
                                   parity);
        parity ^= 1;
        if (W.hi > 0.f) {
          c = cn;
          M = W.hi + W.lo;
          ++nres;
          held = true;
        } else {
          flags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
          held = false;
        }
      }
      if (next < 0) {
        // every child rejected, or a leaf: draw from the held distribution
        if (!held) {
          if (sr.staged && loaded != cur) {
            walk_prefetch<TE>(sr, buf, gp, gq, c > 0.f && !dq.onehot, V);
            loaded = cur;
          }
          walk_pass<TE>(ws, cluster, sr, C, rank, tot, buf, gp, gq, dp, dq, c, V, parity);
          parity ^= 1;
        }
        if (rank != 0) return;  // no remote access follows
        const int residual = c > 0.f ? 1 : 0;
        RowDesc dqc = dq;
        if (residual && !dq.onehot) dqc.invS = dq.invS * c;
        if (tid < kDThreads)
          step_search<TE, false>(sh, tot, nsteps, gp, gq, dp, dqc, residual, V, ws.cud[cur]);
        __syncthreads();
        int token = sh.token;
        if (token < 0) token = dp.a;  // no positive weight (not reachable with finite rows)
        const int near = sh.margin < kRefineGuard * (1.f + c) ? 1 : 0;
        walk_outputs(P, ws, tree, depth, token, flags, dp, dq, residual ? c : 0.f,
                     static_cast<float>(sh.W), nk > 0 ? 2 : 0, residual ? nres : 0, near);
        return;
      }
    }
    // the accepted child is the next node (every thread has read this node's
    // shared state before warp 0 rewrites it)
    ++depth;
    cur = next;
    if (tid == 0) ws.path[depth] = cur;
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

// Launch with programmatic stream serialisation (the kernel may begin while
// the previous one drains; it waits in grid_dependency_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// Launch with clusters of C CTAs and programmatic stream serialisation (the
// kernel may begin while the previous one drains; it waits in
// grid_dependency_wait).
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster_pdl(void (*kern)(KArgs...), int blocks, int threads, int C,
                               size_t smem, cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

// The largest cluster size (`want`, halved while it cannot be scheduled) of
// a kernel with `smem` bytes of dynamic shared memory, cached per device and
// size under a lock shared by every host thread.
struct ClusterCache {
  std::mutex mu;
  int dev = -1;
  size_t smem = 0;
  int C = 0;
};

template <typename... KArgs>
cudaError_t cluster_size(ClusterCache &c, void (*kern)(KArgs...), int threads, int want,
                         size_t smem, int &C) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(c.mu);
  if (dev != c.dev || smem != c.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (want > 8) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
    }
    int size = want;
    for (; size > 1; size /= 2) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(static_cast<unsigned>(size), 1, 1);
      cfg.blockDim = dim3(static_cast<unsigned>(threads), 1, 1);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = static_cast<unsigned>(size);
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n > 0) break;
    }
    c.C = size;
    c.dev = dev;
    c.smem = smem;
  }
  C = c.C;
  return cudaSuccess;
}

// Events a benchmark asked to be recorded around the rows kernel (both set
// or both null; see spec_set_profile_events).
std::mutex g_prof_mu;
cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

template <typename TE>
cudaError_t launch_chain_t(const Params &P, const Exp2Table &tab, size_t smem,
                           cudaStream_t stream) {
  cudaEvent_t prof_start, prof_stop;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    prof_start = g_prof_start;
    prof_stop = g_prof_stop;
  }
  static ClusterCache draw_cache, fdraw_cache, precise_cache;
  const size_t dsmem = (static_cast<size_t>(P.steps) * sizeof(float) + 15) / 16 * 16 +
                       kDrawRecords * sizeof(unsigned long long);
  const size_t psmem = static_cast<size_t>(P.steps) * 2 * sizeof(float2);
  int Cd = 1, Cp = 1;
  const bool filt = P.bmax != nullptr;
  cudaError_t e = filt ? cluster_size(fdraw_cache, chain_draw_kernel<TE, true>, kDThreads,
                                      kDrawCluster, dsmem, Cd)
                       : cluster_size(draw_cache, chain_draw_kernel<TE, false>, kDThreads,
                                      kDrawCluster, dsmem, Cd);
  if (e != cudaSuccess) return e;
  e = cluster_size(precise_cache, chain_precise_kernel<TE>, kPThreads, kPreciseCluster, psmem, Cp);
  if (e != cudaSuccess) return e;
  Cd = std::max(1, std::min(Cd, P.steps));
  Cp = std::max(1, std::min(Cp, P.steps));
  if (prof_start) {
    e = cudaEventRecord(prof_start, stream);
    if (e != cudaSuccess) return e;
  }
  e = launch_chain_rows(P, sizeof(TE), smem, stream, false);
  if (e != cudaSuccess) return e;
  if (prof_stop) {
    e = cudaEventRecord(prof_stop, stream);
    if (e != cudaSuccess) return e;
  }
  if (filt) {  // a row filter: thresholds and kept normalisers first
    e = launch_pdl(chain_filter_kernel<TE>, dim3(static_cast<unsigned>(P.nseq) * (2 * P.gamma + 1)),
                   dim3(kFThreads), 0, stream, P);
    if (e != cudaSuccess) return e;
  }
  e = filt ? launch_cluster_pdl(chain_draw_kernel<TE, true>, P.nseq * Cd, kDThreads, Cd, dsmem,
                                stream, P)
           : launch_cluster_pdl(chain_draw_kernel<TE, false>, P.nseq * Cd, kDThreads, Cd, dsmem,
                                stream, P);
  if (e != cudaSuccess) return e;
  const int gy = std::min(P.nseq, kPreciseGrid);
  return launch_cluster_pdl(chain_precise_kernel<TE>, gy * Cp, kPThreads, Cp, psmem, stream, P,
                            tab);
}

// Staging buffer of a walk CTA: its share of both rows for clusters of C CTAs
// when that fits in kWalkMaxBuf bytes, and at least the records' staging area.
constexpr int kWalkMaxBuf = 96 * 1024;
int walk_buf_bytes(const Params &P, int esize, int C) {
  const long long share = static_cast<long long>((P.steps + C - 1) / C) * kStep * esize * 2;
  const long long recs = static_cast<long long>(kDrawRecords) * sizeof(unsigned long long);
  return static_cast<int>(share <= kWalkMaxBuf ? std::max(share, recs) : recs);
}

template <typename TE>
cudaError_t launch_tree_walk_t(const Params &P, size_t smem, cudaStream_t stream) {
  static ClusterCache walk_cache;
  Params Pw = P;
  Pw.walk_buf = walk_buf_bytes(P, sizeof(TE), kWalkCluster);
  const size_t wsmem = (static_cast<size_t>(P.steps) * sizeof(float) + 15) / 16 * 16 +
                       static_cast<size_t>(Pw.walk_buf);
  int Cw = 1;
  cudaError_t e =
      cluster_size(walk_cache, tree_walk_kernel<TE>, kWThreads, kWalkCluster, wsmem, Cw);
  if (e != cudaSuccess) return e;
  // a smaller cluster whose shares do not fit reads the rows from global memory
  Cw = std::max(1, std::min(Cw, P.steps));
  e = launch_chain_rows(P, sizeof(TE), smem, stream, true);  // behind the first-child kernel
  if (e != cudaSuccess) return e;
  return launch_cluster_pdl(tree_walk_kernel<TE>, P.nseq * Cw, kWThreads, Cw, wsmem, stream, Pw);
}

}  // namespace

bool set_profile_events(void *start, void *stop) {
  if ((start == nullptr) != (stop == nullptr)) return false;
  std::lock_guard<std::mutex> lock(g_prof_mu);
  g_prof_start = static_cast<cudaEvent_t>(start);
  g_prof_stop = static_cast<cudaEvent_t>(stop);
  return true;
}

cudaError_t launch_chain(const Params &P, int esize, const Exp2Table &tab, size_t smem,
                         cudaStream_t stream) {
  return esize == 2 ? launch_chain_t<uint16_t>(P, tab, smem, stream)
                    : launch_chain_t<float>(P, tab, smem, stream);
}

cudaError_t launch_tree_walk(const Params &P, int esize, size_t smem, cudaStream_t stream) {
  return esize == 2 ? launch_tree_walk_t<uint16_t>(P, smem, stream)
                    : launch_tree_walk_t<float>(P, smem, stream);
}

}  // namespace sv
