// Chain verification as four stream-ordered kernels (rows 16-byte aligned,
// no top-k, gamma <= 31).
//
// No kernel here waits on another CTA's progress.  Hand-offs between CTAs are
// kernel boundaries, plus one per-sequence arrival counter in the weights
// kernel: each slice stores its totals, fences (release), and adds one to the
// counter; the slice whose add completes the count fences again (acquire) and
// searches.
//
//  1. rows kernel (the HBM stream).  Every logit row of the batch - the
//     gamma + 1 target rows and the gamma draft rows of each sequence - is cut
//     into 32 KB chunks, numbered sequence-major and handed out round-robin
//     over a persistent grid.  In each CTA one producer warp streams its chunks
//     into a ring of shared-memory slots with bulk asynchronous copies
//     (cp.async.bulk, one "full" and one "empty" mbarrier per slot); eight
//     consumer warps reduce each chunk to one 64-bit record per warp: the
//     (max, sum of 2^((z - max) k)) of a sampling row, k = log2(e) / T, or the
//     (finite max, lowest index + 1) of a greedy row.  Every logit is read from
//     HBM once and costs one exponential; nothing else happens on this path.
//  2. decide kernel, one CTA per sequence: a warp per row merges the row's
//     records into its softmax normaliser (or argmax); one warp then runs the
//     acceptance tests of all gamma positions at once (u < min(1, p/q), one
//     lane each, Philox uniforms), finds the first rejection j with a ballot,
//     and either writes the outputs (a one-hot draw needs no weights) or leaves
//     the draw's description.
//  3. weights kernel, persistent: work items are (sequence, slice); a producer
//     warp copies the slice of the draw row(s) into a ring of shared-memory
//     slots, eight warps sum the draw weights per 256-entry step ([p_j - q_j]_+
//     for a correction, p_gamma for the bonus).  The last slice of a sequence
//     to finish finds the step holding u * W by a prefix over the step totals,
//     scans it, and writes the outputs.  A draw that lands within the
//     single-precision error bound of a CDF boundary is queued.
//  4. precise kernel.  Each queued draw is recomputed with double-float
//     weights, split into pj jobs over its steps; the last job of a draw
//     searches and overwrites the token.
//
// Exponent arithmetic: 2^((z - m) k) with z - m computed exactly (one rounding
// in the product), in the records, the merge, the acceptance test and the draw
// alike, so the normalisers and the draw weights share their scale.
#include <mutex>

#include "ops.cuh"
#include "precise_row.cuh"

namespace sv {

cudaError_t launch_chain_rows(const Params &P, int esize, size_t smem, cudaStream_t stream);

namespace {

constexpr int kKWarps = 16;                            // decide kernel
constexpr int kKThreads = kKWarps * 32;
constexpr int kWWarps = 8;                             // weights kernel: compute warps
constexpr int kWThreads = (kWWarps + 1) * 32;          // + the producer warp
constexpr int kWRing = 4;
constexpr int kDWarps = kWWarps;
constexpr int kDThreads = kWWarps * 32;                // threads of a search
constexpr int kQThreads = 128;                         // precise kernel
constexpr int kQWarps = kQThreads / 32;
constexpr int kStep = 256;  // entries per draw-search step
constexpr int kCMaxGamma = 31;
constexpr int kCMaxRows = 2 * kCMaxGamma + 1;
constexpr uint32_t kNoIndex = 0x3FFFFFFFu;  // record index: no finite entry
constexpr uint32_t kBadBit = 0x80000000u;   // record index bit: NaN or +inf seen

__device__ __forceinline__ void mbar_arrive1_c(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

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
__device__ __forceinline__ Df ld_df(const float2 *p) {
  const float2 v = __ldcg(p);
  return Df{v.x, v.y};
}
// from shared memory when staged, else from global memory
__device__ __forceinline__ Df ld_dfs(const float2 *p, bool staged) {
  if (staged) return Df{p->x, p->y};
  return ld_df(p);
}

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

// Barrier over the compute warps of the weights kernel (named barrier 1).
__device__ __forceinline__ void wsync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

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
// 2. decide kernel
// ---------------------------------------------------------------------------

// 2^((z - m) k): the exponent form every step of the chain path uses.
__device__ __forceinline__ float pexp(float z, float m, float k) {
  return fast_exp2(__fmul_rn(__fsub_rn(z, m), k));
}

// Probability of entry v with logit z under a row descriptor.
__device__ __forceinline__ float pprob(const RowDesc &d, float z, int v) {
  if (d.onehot) return v == d.a ? 1.f : 0.f;
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

// The merged record of row r of sequence seq (one warp; the value in every
// lane): the rows kernel stored all of the row's records before this kernel.
__device__ unsigned long long merge_row(const Params &P, int seq, int r) {
  const int lane = threadIdx.x & 31;
  const int rps = 2 * P.gamma + 1;
  const bool draft = r > P.gamma;
  const float T = __ldg((draft ? P.Tq : P.Tp) + seq);
  const bool arg = row_is_arg(T);
  const float k = arg ? 0.f : kLog2e / T;
  const int R = P.cpr * kChainRecordsPerChunk;
  const unsigned long long *rec =
      P.srec + (static_cast<long long>(seq) * rps + r) * static_cast<long long>(R);
  float m = -INFINITY, S = 0.f, bv = -INFINITY;
  uint32_t bi = kNoIndex;
  int bad = 0;
  for (int x0 = lane; x0 < R; x0 += 4 * 32) {
    unsigned long long b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) b[i] = x0 + i * 32 < R ? __ldcg(rec + x0 + i * 32) : 0ull;
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

// Decide sequence seq from its rows' records (one warp): the acceptance
// tests, the first rejection j, and either the outputs (a one-hot draw needs
// no weights) or the draw's description for the weights kernel.
template <typename TE>
__device__ void decide_seq(const Params &P, int seq, const unsigned long long *rr) {
  const int lane = threadIdx.x & 31;
  const int gamma = P.gamma, V = P.V;
  const float Tp = __ldg(P.Tp + seq), Tq = __ldg(P.Tq + seq);
  const bool p_arg = row_is_arg(Tp), q_arg = row_is_arg(Tq);
  const bool tp_bad = !(Tp >= 0.f) || Tp == INFINITY, tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  const float kp = p_arg ? 0.f : kLog2e / Tp, kq = q_arg ? 0.f : kLog2e / Tq;
  // lane i holds target row i (i <= gamma) and draft row gamma + 1 + i (i < gamma)
  const int i = lane;
  RowDesc dp = row_desc(i <= gamma ? rr[i] : 0ull, p_arg, tp_bad, kp, V);
  RowDesc dq = row_desc(i < gamma ? rr[gamma + 1 + i] : 0ull, q_arg, tq_bad, kq, V);
  // rows whose sampling statistics were not finite: the finite argmax (rare)
  unsigned need = __ballot_sync(0xFFFFFFFFu, i <= gamma && !p_arg && dp.onehot);
  while (need) {
    const int src = __ffs(need) - 1;
    need &= need - 1;
    const int a = warp_finite_argmax<TE>(chain_row<TE>(P, seq, src), V);
    if (lane == src) dp.a = a;
  }
  need = __ballot_sync(0xFFFFFFFFu, i < gamma && !q_arg && dq.onehot);
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
    const int x = __ldg(P.tokens + static_cast<long long>(seq) * gamma + i);
    f = dp.flags;
    const bool valid = x >= 0 && x < V;
    if (!valid) f |= SPEC_FLAG_BAD_TOKEN;
    if (dp.onehot) {
      reject = !(valid && x == dp.a);
    } else {
      f |= dq.flags;
      if (valid) {
        const TE *gp = chain_row<TE>(P, seq, i);
        const TE *gq = chain_row<TE>(P, seq, gamma + 1 + i);
        const float px = pprob(dp, to_f32(gp[x]), x);
        const float qx = pprob(dq, dq.onehot ? 0.f : to_f32(gq[x]), x);
        if (!(qx > 0.f)) {
          f |= SPEC_FLAG_ZERO_Q;
        } else {
          const float uu = unit_uniform(P, seq, i, 0);
          reject = !(uu < fminf(1.f, px / qx));
        }
      }
    }
  }
  const unsigned rej = __ballot_sync(0xFFFFFFFFu, reject && i < gamma);
  const int j = rej ? __ffs(rej) - 1 : gamma;
  const float ud = i <= gamma ? unit_uniform(P, seq, i, 1) : 0.f;
  const float u_draw = __shfl_sync(0xFFFFFFFFu, ud, j);
  uint32_t fo = warp_or(i < j ? f : 0u);
  fo |= __shfl_sync(0xFFFFFFFFu, i < gamma ? f : dp.flags, j);  // position j's flags
  const RowDesc djp = shfl_desc(dp, j);
  const RowDesc djq = shfl_desc(dq, j);
  if (lane == 0 && __ldcg(P.err)) {
    // a bounded wait of the rows kernel gave up: the documented fallback, no
    // accepted drafts and no tokens
    const long long obase = static_cast<long long>(seq) * (gamma + 1);
    for (int x = 0; x <= gamma; ++x) P.out_tokens[obase + x] = -1;
    P.out_num[seq] = 0;
    if (P.out_flags) P.out_flags[seq] = SPEC_FLAG_TIMEOUT;
    P.final_unit[seq] = -1;
    PassSeq ps = {};
    ps.draw = 0;
    reinterpret_cast<PassSeq *>(P.pseqw)[seq] = ps;
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
      write_outputs(P, seq, ps, ps.dp.a, 0.0, 0);
    }
    reinterpret_cast<PassSeq *>(P.pseqw)[seq] = ps;  // read by the weights kernel
  }
}

// One CTA per sequence: a warp per row merges, warp 0 decides.
template <typename TE>
__global__ void __launch_bounds__(kKThreads) chain_decide_kernel(const Params P) {
  __shared__ unsigned long long rr[kCMaxRows];
  launch_dependents();
  grid_dependency_wait();
  const int seq = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rps = 2 * P.gamma + 1;
  for (int r = warp; r < rps; r += kKWarps) {
    const unsigned long long rec = merge_row(P, seq, r);
    if (lane == 0) rr[r] = rec;
  }
  __syncthreads();
  if (warp == 0) decide_seq<TE>(P, seq, rr);
}

// ---------------------------------------------------------------------------
// 3. weights kernel
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
// rows use packed pairs, rounding exactly like pprob().
__device__ __forceinline__ void weights8(const RowDesc &dp, const RowDesc &dq, int residual,
                                         int base, const float zp[8], const float zq[8],
                                         float w[8]) {
  if (!dp.onehot && (!residual || !dq.onehot)) {
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
    float x = pprob(dp, zp[e], base + e);
    if (residual) x = fmaxf(x - pprob(dq, zq[e], base + e), 0.f);
    w[e] = x;
  }
}

// Draw weights of 8 entries from `base` (entries at or past V are 0).
template <typename TE>
__device__ __forceinline__ void step_weights(const TE *gp, const TE *gq, const RowDesc &dp,
                                             const RowDesc &dq, int residual, int base, int V,
                                             float w[8]) {
  float zp[8], zq[8];
  const bool full = base + 8 <= V;
  if (full && !dp.onehot) {
    load_vec<TE>(gp + base, zp);
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) zp[e] = (!dp.onehot && base + e < V) ? to_f32(gp[base + e]) : 0.f;
  }
  if (residual) {
    if (full && !dq.onehot) {
      load_vec<TE>(gq + base, zq);
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e)
        zq[e] = (!dq.onehot && base + e < V) ? to_f32(gq[base + e]) : 0.f;
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) zq[e] = 0.f;
  }
  weights8(dp, dq, residual, base, zp, zq, w);  // the same arithmetic as the records
#pragma unroll
  for (int e = 0; e < 8; ++e)
    if (base + e >= V) w[e] = 0.f;
}

// Totals of the draw weights of steps [b0, b1) (256 entries each) into
// fst[step] (the whole CTA, one warp per step; full steps four per warp at a
// time with their loads issued before any is used).
template <typename TE>
__device__ void step_totals(const TE *gp, const TE *gq, const RowDesc &dp, const RowDesc &dq,
                            int residual, int V, int b0, int b1, float *fst) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  constexpr int kU = 4;
  const int nfull = min(b1, V / kStep);
  int st0 = b0 + w;
  if (!dp.onehot && (!residual || !dq.onehot)) {
    for (; st0 + (kU - 1) * kDWarps < nfull; st0 += kDWarps * kU) {
      Raw8<TE> rp[kU], rq[kU];
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int base = (st0 + q * kDWarps) * kStep + lane * 8;
        rp[q].load(gp + base);
        if (residual) rq[q].load(gq + base);
      }
#pragma unroll
      for (int q = 0; q < kU; ++q) {
        const int base = (st0 + q * kDWarps) * kStep + lane * 8;
        float zp[8], zq[8], x[8];
        rp[q].get(zp);
        rq[q].get(zq);
        weights8(dp, dq, residual, base, zp, zq, x);
        float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
        sm = warp_sum(sm);
        if (lane == 0) fst[st0 + q * kDWarps] = sm;
      }
    }
  }
  for (int st = st0; st < b1; st += kDWarps) {
    float x[8];
    step_weights<TE>(gp, gq, dp, dq, residual, st * kStep + lane * 8, V, x);
    float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    sm = warp_sum(sm);
    if (lane == 0) fst[st] = sm;
  }
}

// Step totals the draw search stages in shared memory (rows of up to
// kSmemSteps * 256 entries; longer rows are searched from global memory).
constexpr int kSmemSteps = 2048;

struct DrawCtl {
  double W;
  int token;
  float margin;
  int is_last;
  float tot[kSmemSteps];
};

// Inverse-CDF search over the step totals fst[0, nsteps) (the compute warps;
// warp 0 works): a double-float prefix over the lanes' runs of steps finds the
// step holding u * W, one warp scan of its weights the token.  The token goes
// to ctl.token (-1: no positive weight), the total to ctl.W and the distance
// of the draw from the nearer boundary of its token to ctl.margin.
template <typename TE>
__device__ void step_search(DrawCtl &ctl, const float *gst, int nsteps, const TE *gp,
                            const TE *gq, const RowDesc &dp, const RowDesc &dq, int residual,
                            int V, float u) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  // the totals in one coalesced pass
  const bool staged = nsteps <= kSmemSteps;
  if (staged)
    for (int st0 = threadIdx.x; st0 < nsteps; st0 += 4 * kDThreads) {  // four loads in flight
      float x[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) x[q] = st0 + q * kDThreads < nsteps ? __ldcg(gst + st0 + q * kDThreads) : 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (st0 + q * kDThreads < nsteps) ctl.tot[st0 + q * kDThreads] = x[q];
    }
  wsync();
  const float *fst = staged ? ctl.tot : gst;
  if (w == 0) {
    const int per = (nsteps + 31) / 32;
    const int s0 = min(nsteps, lane * per), s1 = min(nsteps, s0 + per);
    Df seg{0.f, 0.f};
    int lastpos = -1;
    for (int st = s0; st < s1; ++st) {
      const float x = staged ? fst[st] : __ldcg(fst + st);
      seg = df_add(seg, Df{x, 0.f});
      if (x > 0.f) lastpos = st;
    }
    Df incl = seg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const Df y = df_shfl_up(incl, off);
      if (lane >= off) incl = df_add(incl, y);
    }
    const Df W = df_shfl(incl, 31);
    const Df tt = df_mul(Df{u, 0.f}, W);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, df_gt(incl, tt) && seg.hi > 0.f);
    int step = -1;
    float trel = 0.f;
    bool exact = true;
    if (hit) {
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        Df acc = df_sub(incl, seg);
        for (int st = s0; st < s1; ++st) {
          const float x = staged ? fst[st] : __ldcg(fst + st);
          const Df nx = df_add(acc, Df{x, 0.f});
          if (df_gt(nx, tt) && x > 0.f) {
            step = st;
            const Df r = df_sub(tt, acc);
            trel = r.hi + r.lo;
            break;
          }
          acc = nx;
        }
        if (step < 0) {
          step = lastpos;
          exact = false;
        }
      }
      step = __shfl_sync(0xFFFFFFFFu, step, first);
      trel = __shfl_sync(0xFFFFFFFFu, trel, first);
      exact = __shfl_sync(0xFFFFFFFFu, exact ? 1 : 0, first) != 0;
    } else {
      step = warp_max_i(lastpos);
      exact = false;
    }
    int token = -1;
    float margin = 0.f;
    if (step >= 0) {
      const float tr = trel;
      const int base = step * kStep + lane * 8;
      float x[8];
      step_weights<TE>(gp, gq, dp, dq, residual, base, V, x);
      float sm = 0.f;
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sm += x[e];
        if (x[e] > 0.f) lp = base + e;
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
        const int first = __ffs(h2) - 1;
        int found = -1;
        float mg = 0.f;
        if (lane == first) {
          float run = excl;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float prev = run;
            run += x[e];
            if (found < 0 && x[e] > 0.f && run > tr) {
              found = base + e;
              mg = fminf(tr - prev, run - tr);
            }
          }
          if (found < 0) found = lp;
        }
        token = __shfl_sync(0xFFFFFFFFu, found, first);
        margin = __shfl_sync(0xFFFFFFFFu, mg, first);
      } else {
        token = warp_max_i(lp);
        margin = 0.f;
      }
    }
    if (lane == 0) {
      ctl.W = static_cast<double>(W.hi) + static_cast<double>(W.lo);
      ctl.token = token;
      ctl.margin = margin;
    }
  }
  wsync();
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

// One work item of the weights kernel in a ring slot: a slice of a draw's
// row(s), with the draw's description.
struct WItem {
  PassSeq ps;
  int seq;
  int b0, b1;  // steps of the slice
  int nb;      // entries of the slice copied to shared memory (the rest: global)
  int pad[3];
};

struct WCtl {
  unsigned long long full[kWRing];
  unsigned long long empty[kWRing];
  WItem item[kWRing];
};

// Totals of the draw weights of the slice's steps from the slot (entries past
// nb, fewer than 8 at the row's end, from global memory) into fst[step].
template <typename TE>
__device__ void slot_step_totals(const TE *sp, const TE *sq, const TE *gp, const TE *gq,
                                 const WItem &it, int V, float *fst) {
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const PassSeq &ps = it.ps;
  const int v0 = it.b0 * kStep;
  for (int st = it.b0 + w; st < it.b1; st += kWWarps) {
    const int base = st * kStep + lane * 8;  // vocabulary index
    const int e = base - v0;                 // slot index
    float x[8];
    if (e + 8 <= it.nb && !ps.dp.onehot && (!ps.residual || !ps.dq.onehot)) {
      float zp[8], zq[8];
      load_vec<TE>(sp + e, zp);
      if (ps.residual) load_vec<TE>(sq + e, zq);
      else
#pragma unroll
        for (int q = 0; q < 8; ++q) zq[q] = 0.f;
      weights8(ps.dp, ps.dq, ps.residual, base, zp, zq, x);
    } else {
      step_weights<TE>(gp, gq, ps.dp, ps.dq, ps.residual, base, V, x);
    }
    float sm = ((x[0] + x[1]) + (x[2] + x[3])) + ((x[4] + x[5]) + (x[6] + x[7]));
    sm = warp_sum(sm);
    if (lane == 0) fst[st] = sm;
  }
}

// Persistent: item k (sequence k / wj, slice k % wj) goes to CTA k mod grid.
template <typename TE>
__global__ void __launch_bounds__(kWThreads) chain_weights_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  WCtl &ctl = *reinterpret_cast<WCtl *>(smem_raw);
  unsigned char *ring = smem_raw + P.data_off;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int V = P.V, nsteps = P.steps, S = P.wj;
  const long long total = static_cast<long long>(P.nseq) * S;
  const int slot_bytes = P.slot_bytes;  // one slice of one row
  launch_dependents();
  grid_dependency_wait();
  if (threadIdx.x == 0) {
    for (int s = 0; s < kWRing; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], kWWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();
  if (warp == kWWarps) {
    // producer: the item's description, then bulk copies of its slice; the
    // next item's description is loaded while this one's slot is awaited
    if (lane != 0) return;
    int i = 0;
    long long k = blockIdx.x;
    PassSeq nxt;
    if (k < total) nxt = reinterpret_cast<const PassSeq *>(P.pseqw)[k / S];
    for (; k < total; k += gridDim.x, ++i) {
      const PassSeq cur = nxt;
      if (k + gridDim.x < total) nxt = reinterpret_cast<const PassSeq *>(P.pseqw)[(k + gridDim.x) / S];
      const int slot = i % kWRing;
      if (i >= kWRing) {
        const uint32_t ph = static_cast<uint32_t>((i - kWRing) / kWRing) & 1u;
        if (!mbar_wait_bounded(&ctl.empty[slot], ph)) atomicOr(P.err, 1u);
      }
      WItem &it = ctl.item[slot];
      it.seq = static_cast<int>(k / S);
      const int s = static_cast<int>(k - static_cast<long long>(it.seq) * S);
      it.ps = cur;
      it.b0 = s * P.wj_steps;
      it.b1 = min(nsteps, it.b0 + P.wj_steps);
      uint32_t bytes = 0u;
      it.nb = 0;
      if (cur.draw && it.b0 < it.b1) {
        const TE *gp, *gq;
        draw_rows<TE>(P, it.seq, cur.j, gp, gq);
        const int v0 = it.b0 * kStep, v1 = min(V, it.b1 * kStep);
        const uint32_t rb = static_cast<uint32_t>((v1 - v0) * sizeof(TE)) / 16u * 16u;
        it.nb = static_cast<int>(rb / sizeof(TE));
        unsigned char *dst = ring + static_cast<size_t>(slot) * 2 * slot_bytes;
        bytes = cur.residual ? 2u * rb : rb;
        mbar_arrive_expect_tx(&ctl.full[slot], bytes);
        if (rb) {
          bulk_g2s_plain(dst, gp + v0, rb, &ctl.full[slot]);
          if (cur.residual) bulk_g2s_plain(dst + slot_bytes, gq + v0, rb, &ctl.full[slot]);
        }
      } else {
        mbar_arrive_expect_tx(&ctl.full[slot], 0u);
      }
    }
    const int issued = i;
    for (int d = max(0, issued - kWRing); d < issued; ++d) {
      const uint32_t ph = static_cast<uint32_t>(d / kWRing) & 1u;
      if (!mbar_wait_bounded(&ctl.empty[d % kWRing], ph)) atomicOr(P.err, 1u);
    }
    return;
  }
  int i = 0;
  for (long long k = blockIdx.x; k < total; k += gridDim.x, ++i) {
    const int slot = i % kWRing;
    const uint32_t phase = static_cast<uint32_t>(i / kWRing) & 1u;
    if (!mbar_wait_bounded(&ctl.full[slot], phase)) {
      if (lane == 0) atomicOr(P.err, 1u);
      mbar_wait_bounded(&ctl.full[slot], phase);  // do not leave a copy in flight
    }
    const WItem it = ctl.item[slot];
    const int seq = it.seq;
    const bool work = it.ps.draw && it.b0 < it.b1;
    float *fst = reinterpret_cast<float *>(P.fstep) + static_cast<long long>(seq) * nsteps;
    const TE *gp, *gq;
    draw_rows<TE>(P, seq, it.ps.j, gp, gq);
    if (work) {
      const TE *sp = reinterpret_cast<const TE *>(ring + static_cast<size_t>(slot) * 2 * slot_bytes);
      const TE *sq = reinterpret_cast<const TE *>(ring + static_cast<size_t>(slot) * 2 * slot_bytes +
                                                  slot_bytes);
      slot_step_totals<TE>(sp, sq, gp, gq, it, V, fst);
    }
    __syncwarp();
    if (lane == 0) mbar_arrive1_c(&ctl.empty[slot]);  // the slot's data is no longer read
  }
}

// One CTA per sequence, after the weights kernel: the inverse-CDF search over
// the draw's step totals, the outputs, and the queue of draws for the precise
// redraw.
template <typename TE>
__global__ void __launch_bounds__(kDThreads) chain_search_kernel(const Params P) {
  __shared__ DrawCtl ctl;
  launch_dependents();
  grid_dependency_wait();
  const int seq = blockIdx.x;
  PassSeq ps = reinterpret_cast<const PassSeq *>(P.pseqw)[seq];
  if (!ps.draw) return;  // the decide kernel wrote the outputs
  if (__ldcg(P.err)) {
    // a bounded wait of the weights kernel gave up: the step totals may be
    // incomplete, so the draw gets the fallback outputs
    if (threadIdx.x == 0) {
      const long long obase = static_cast<long long>(seq) * (P.gamma + 1);
      for (int x = 0; x <= P.gamma; ++x) P.out_tokens[obase + x] = -1;
      P.out_num[seq] = 0;
      if (P.out_flags) P.out_flags[seq] = SPEC_FLAG_TIMEOUT;
      P.final_unit[seq] = -1;
    }
    return;
  }
  const int V = P.V, nsteps = P.steps;
  float *fst = reinterpret_cast<float *>(P.fstep) + static_cast<long long>(seq) * nsteps;
  const TE *gp, *gq;
  draw_rows<TE>(P, seq, ps.j, gp, gq);
  step_search<TE>(ctl, fst, nsteps, gp, gq, ps.dp, ps.dq, ps.residual, V, ps.u);
  int token = ctl.token;
  double W = ctl.W;
  float margin = ctl.margin;
  if (ps.residual && !(W > 0.0)) {
    // degenerate residual: draw from p itself
    ps.flags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
    ps.residual = 0;
    ps.dq = ps.dp;
    ps.dq.onehot = 1;
    ps.dq.a = 0;
    wsync();
    step_totals<TE>(gp, gq, ps.dp, ps.dq, 0, V, 0, nsteps, fst);
    wsync();
    step_search<TE>(ctl, fst, nsteps, gp, gq, ps.dp, ps.dq, 0, V, ps.u);
    token = ctl.token;
    W = ctl.W;
    margin = ctl.margin;
  }
  if (token < 0) token = ps.dp.a;  // no positive weight at all (not reachable with finite rows)
  // redraw precisely when the draw came within 1e-6 of the draw mass of a
  // boundary (the single-precision boundary error measured on 128K-entry rows
  // stays below 3e-7 of it)
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
// 3. precise kernel
// ---------------------------------------------------------------------------

// Step sums the precise search stages in shared memory (rows of up to
// kQSmemSteps * 256 entries; longer rows are searched from global memory).
constexpr int kQSmemSteps = 2048;

struct QCtl {
  float tab_hi[64], tab_lo[64];
  Df pred[2][kQWarps];
  int red_i[kQWarps];
  int redo;
  float2 sa[kQSmemSteps], sb[kQSmemSteps];
};

// Double-float weights of the 8 entries from `base` (precise redraw).
template <typename TE>
__device__ __forceinline__ void pweights8(const TE *gp, const TE *gq, const HpRow &rp,
                                          const HpRow &rq, int residual, Df rho, int base, int V,
                                          bool vec, const QCtl &ctl, Df w[8]) {
  float zp[8], zq[8];
  hp_load8<TE>(gp, base, V, vec, zp);
  if (residual) hp_load8<TE>(gq, base, V, vec, zq);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const Df ep = hp_exp(rp, zp[e], ctl.tab_hi, ctl.tab_lo);
    if (!residual || ep.hi == 0.f) {
      w[e] = ep;
      continue;
    }
    const Df eq = hp_exp(rq, zq[e], ctl.tab_hi, ctl.tab_lo);
    const Df d = df_sub(ep, df_mul(rho, eq));
    w[e] = d.hi > 0.f ? d : Df{0.f, 0.f};
  }
}

// Sum over the pj normaliser shares of sequence s (the same value in every
// lane: lane-strided sums, a butterfly).
__device__ __forceinline__ Df pshare_sum(const Params &P, int s, int which) {
  const int lane = threadIdx.x & 31;
  const float2 *x = reinterpret_cast<const float2 *>(P.ppart) + static_cast<long long>(s) * P.pj * 2 + which;
  Df v{0.f, 0.f};
  for (int k0 = 0; k0 < P.pj; k0 += 64) {  // two loads in flight per lane
    const int ka = k0 + lane, kb = k0 + 32 + lane;
    const Df a = ka < P.pj ? ld_df(x + 2 * ka) : Df{0.f, 0.f};
    const Df b = kb < P.pj ? ld_df(x + 2 * kb) : Df{0.f, 0.f};
    v = df_add(v, df_add(a, b));
  }
  return df_warp_sum(v);
}

// Search of a precise redraw (the CTA that completed the draw's jobs).  The
// step totals are A - rho B with rho = S_p / S_q from the normaliser shares (A
// alone for a draw from p); steps a job marked uncertain are first recomputed
// entry by entry.  One warp then finds the step by a prefix over its lanes'
// runs of steps and scans it with double-float weights; the token is
// overwritten.  All sums are double-float (about 48 significant bits).
template <typename TE>
__device__ void psearch(const Params &P, QCtl &ctl, int s, const PassSeq &ps, const TE *gp,
                        const TE *gq, const HpRow &rp, const HpRow &rq, bool vec) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int nsteps = P.steps;
  float2 *pa = reinterpret_cast<float2 *>(P.pstep) + static_cast<long long>(s) * 2 * nsteps;
  float2 *pb = pa + nsteps;
  Df rho{0.f, 0.f};
  if (ps.residual) {
    const Df Sp = pshare_sum(P, s, 0), Sq = pshare_sum(P, s, 1);
    // rho = Sp / Sq as a double-float: q1 = Sp.hi / Sq.hi, then one correction
    // step q2 = (Sp - q1 Sq) / Sq.hi
    const float q1 = __fdiv_rn(Sp.hi, Sq.hi);
    const Df r = df_sub(Sp, df_mul(Df{q1, 0.f}, Sq));
    const float q2 = __fdiv_rn(r.hi, Sq.hi);
    rho = df_norm(q1, q2);
  }
  if (t == 0) ctl.redo = static_cast<int>(__ldcg(P.sctr + 4ll * s + 3));
  __syncthreads();
  if (ctl.redo) {
    // uncertain steps (B < 0): their exact totals, one warp per step
    for (int base = w * 32; base < nsteps; base += kQWarps * 32) {
      const int st = base + lane;
      unsigned todo = __ballot_sync(0xFFFFFFFFu, st < nsteps && __ldcg(&pb[st].x) < 0.f);
      while (todo) {
        const int x = base + __ffs(todo) - 1;
        todo &= todo - 1;
        Df wd[8];
        pweights8<TE>(gp, gq, rp, rq, ps.residual, rho, x * kStep + lane * 8, P.V, vec, ctl, wd);
        Df acc{0.f, 0.f};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc = df_add(acc, wd[e]);
        acc = df_warp_sum(acc);
        if (lane == 0) {
          pa[x] = make_float2(acc.hi, acc.lo);
          pb[x] = make_float2(0.f, 0.f);
        }
      }
    }
    __threadfence_block();
    __syncthreads();
  }
  // the step sums in one coalesced pass (other CTAs wrote most of them)
  const bool staged = nsteps <= kQSmemSteps;
  if (staged)
    for (int st0 = t; st0 < nsteps; st0 += 4 * kQThreads) {  // eight loads in flight
      float2 xa[4], xb[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int st = st0 + q * kQThreads;
        xa[q] = st < nsteps ? __ldcg(pa + st) : make_float2(0.f, 0.f);
        xb[q] = st < nsteps ? __ldcg(pb + st) : make_float2(0.f, 0.f);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int st = st0 + q * kQThreads;
        if (st < nsteps) {
          ctl.sa[st] = xa[q];
          ctl.sb[st] = xb[q];
        }
      }
    }
  __syncthreads();
  const float2 *qa = staged ? ctl.sa : pa, *qb = staged ? ctl.sb : pb;
  if (w == 0) {
    const int per = (nsteps + 31) / 32;
    const int s0 = min(nsteps, lane * per), s1 = min(nsteps, s0 + per);
    const Df nrho{-rho.hi, -rho.lo};
    Df seg{0.f, 0.f};
    int lastpos = -1;
    for (int st = s0; st < s1; ++st) {
      const Df x = df_add(ld_dfs(qa + st, staged), df_mul(nrho, ld_dfs(qb + st, staged)));
      seg = df_add(seg, x);
      if (x.hi > 0.f) lastpos = st;
    }
    Df incl = seg;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const Df y = df_shfl_up(incl, off);
      if (lane >= off) incl = df_add(incl, y);
    }
    const Df Z = df_shfl(incl, 31);
    const Df tt = df_mul(Df{ps.u, 0.f}, Z);
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, df_gt(incl, tt) && seg.hi > 0.f);
    int step = -1;
    Df trel{0.f, 0.f};
    bool exact = true;
    if (hit) {
      const int first = __ffs(hit) - 1;
      if (lane == first) {
        Df acc = df_sub(incl, seg);
        for (int st = s0; st < s1 && step < 0; ++st) {
          const Df x = df_add(ld_dfs(qa + st, staged), df_mul(nrho, ld_dfs(qb + st, staged)));
          if (df_gt(df_add(acc, x), tt) && x.hi > 0.f) {
            step = st;
            trel = df_sub(tt, acc);
          }
          acc = df_add(acc, x);
        }
        if (step < 0) {
          step = lastpos;
          exact = false;
        }
      }
      step = __shfl_sync(0xFFFFFFFFu, step, first);
      trel = df_shfl(trel, first);
      exact = __shfl_sync(0xFFFFFFFFu, exact ? 1 : 0, first) != 0;
    } else {
      step = warp_max_i(lastpos);
      exact = false;
    }
    int token = -1;
    if (step >= 0) {
      const int base = step * kStep + lane * 8;
      Df wd[8];
      pweights8<TE>(gp, gq, rp, rq, ps.residual, rho, base, P.V, vec, ctl, wd);
      Df sm{0.f, 0.f};
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        sm = df_add(sm, wd[e]);
        if (wd[e].hi > 0.f) lp = base + e;
      }
      Df fin = sm;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const Df y = df_shfl_up(fin, off);
        if (lane >= off) fin = df_add(fin, y);
      }
      const unsigned h2 = exact ? __ballot_sync(0xFFFFFFFFu, df_gt(fin, trel) && sm.hi > 0.f) : 0u;
      if (h2) {
        const int first = __ffs(h2) - 1;
        int found = -1;
        if (lane == first) {
          Df run = df_sub(fin, sm);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            run = df_add(run, wd[e]);
            if (found < 0 && wd[e].hi > 0.f && df_gt(run, trel)) found = base + e;
          }
          if (found < 0) found = lp;
        }
        token = __shfl_sync(0xFFFFFFFFu, found, first);
      } else {
        token = warp_max_i(lp);
      }
    }
    if (lane == 0 && token >= 0) {
      const long long obase = static_cast<long long>(s) * (P.gamma + 1);
      P.out_tokens[obase + ps.j] = token;
      P.outs[obase + ps.j].token = token;
    }
  }
  __syncthreads();
}

// Precise job (item, k): redraw item `item` of the queue, slice k of its
// steps.  For each 256-entry step of the slice it stores the double-float sums
// A of e_p and B of e_q over the entries whose weight e_p - rho e_q is
// certainly positive, classified with the single-precision rho of the row
// statistics (within 1e-6 of the exact one; an entry is certain when
// |e_p - rho e_q| > 1e-5 e_p), or B = -1 when an entry of the step is
// uncertain; and the slice's shares of S_p and S_q.  A draw from p stores
// A = the sum of e_p, B = 0.
template <typename TE>
__device__ void pjob(const Params &P, QCtl &ctl, int item, int k) {
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  const int kp = P.pj;
  const int s = __ldcg(P.near_list + item) - 1;  // written by the draw kernel
  if (s < 0 || s >= P.nseq) return;
  const PassSeq ps = reinterpret_cast<const PassSeq *>(P.pseqw)[s];
  if (ps.j < 0 || ps.j > P.gamma) return;  // not a drawn position: never use it as a row
  const TE *gp, *gq;
  draw_rows<TE>(P, s, ps.j, gp, gq);
  const bool vec = ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(gq)) & 15u) == 0;
  const HpRow rp = hp_row(ps.dp, __ldg(P.Tp + s));
  const HpRow rq = ps.residual ? hp_row(ps.dq, __ldg(P.Tq + s)) : rp;
  const int residual = ps.residual;
  const float rho_a = residual ? ps.dq.invS / ps.dp.invS : 0.f;  // S_p / S_q, single precision
  const int V = P.V;
  const int b0 = k * P.pj_steps, b1 = min(P.steps, b0 + P.pj_steps);
  float2 *pa = reinterpret_cast<float2 *>(P.pstep) + static_cast<long long>(s) * 2 * P.steps;
  float2 *pb = pa + P.steps;
  uint32_t *cnt = P.sctr + 4ll * s;
  Df sp_tot{0.f, 0.f}, sq_tot{0.f, 0.f};
  bool unc_any = false;
  for (int st = b0 + w; st < b1; st += kQWarps) {
    const int base = st * kStep + lane * 8;
    float zp[8], zq[8];
    hp_load8<TE>(gp, base, V, vec, zp);
    if (residual) hp_load8<TE>(gq, base, V, vec, zq);
    Df sp{0.f, 0.f}, sq{0.f, 0.f}, a{0.f, 0.f}, b{0.f, 0.f};
    bool unc = false;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const Df ep = hp_exp(rp, zp[e], ctl.tab_hi, ctl.tab_lo);
      sp = df_add(sp, ep);
      if (!residual) continue;
      const Df eq = hp_exp(rq, zq[e], ctl.tab_hi, ctl.tab_lo);
      sq = df_add(sq, eq);
      if (ep.hi > 0.f) {
        const float d = fmaf(-rho_a, eq.hi, ep.hi);
        if (d > 1e-5f * ep.hi) {
          a = df_add(a, ep);
          b = df_add(b, eq);
        } else if (d >= -1e-5f * ep.hi) {
          unc = true;
        }
      }
    }
    const Df A = df_warp_sum(residual ? a : sp);
    const Df Bq = df_warp_sum(b);
    unc = __any_sync(0xFFFFFFFFu, unc);
    if (lane == 0) {
      pa[st] = make_float2(A.hi, A.lo);
      pb[st] = unc ? make_float2(-1.f, 0.f) : make_float2(Bq.hi, Bq.lo);
    }
    unc_any |= unc;
    sp_tot = df_add(sp_tot, sp);
    sq_tot = df_add(sq_tot, sq);
  }
  sp_tot = df_warp_sum(sp_tot);
  sq_tot = df_warp_sum(sq_tot);
  if (lane == 0) {
    ctl.pred[0][w] = sp_tot;
    ctl.pred[1][w] = sq_tot;
    ctl.red_i[w] = unc_any ? 1 : 0;
  }
  __syncthreads();
  if (t == 0) {
    Df A{0.f, 0.f}, B{0.f, 0.f};
    int u = 0;
    for (int x = 0; x < kQWarps; ++x) {
      A = df_add(A, ctl.pred[0][x]);
      B = df_add(B, ctl.pred[1][x]);
      u |= ctl.red_i[x];
    }
    float2 *dst = reinterpret_cast<float2 *>(P.ppart) + (static_cast<long long>(s) * kp + k) * 2;
    dst[0] = make_float2(A.hi, A.lo);
    dst[1] = make_float2(B.hi, B.lo);
    if (u) atomicAdd(cnt + 3, 1u);  // read by the search kernel, after this one
  }
  __syncthreads();  // ctl.pred is reused by the CTA's next item
}

// Grid (job, item stride): CTA (k, y) runs job k of queued draws
// y, y + gridDim.y, ...
template <typename TE>
__global__ void __launch_bounds__(kQThreads) chain_precise_kernel(const Params P,
                                                                  const Exp2Table tab) {
  __shared__ QCtl ctl;
  launch_dependents();
  grid_dependency_wait();
  const uint32_t count = min(__ldcg(P.pctr), static_cast<uint32_t>(P.nseq));
  if (blockIdx.y >= count) return;
  for (int i = threadIdx.x; i < 64; i += kQThreads) {
    ctl.tab_hi[i] = tab.hi[i];
    ctl.tab_lo[i] = tab.lo[i];
  }
  __syncthreads();
  for (uint32_t item = blockIdx.y; item < count; item += gridDim.y)
    pjob<TE>(P, ctl, static_cast<int>(item), blockIdx.x);
}

// One CTA per queued draw (stride gridDim.x), after the precise jobs: the
// double-float search and the token.
template <typename TE>
__global__ void __launch_bounds__(kQThreads) chain_psearch_kernel(const Params P,
                                                                  const Exp2Table tab) {
  __shared__ QCtl ctl;
  launch_dependents();
  grid_dependency_wait();
  const uint32_t count = min(__ldcg(P.pctr), static_cast<uint32_t>(P.nseq));
  if (blockIdx.x >= count) return;
  for (int i = threadIdx.x; i < 64; i += kQThreads) {
    ctl.tab_hi[i] = tab.hi[i];
    ctl.tab_lo[i] = tab.lo[i];
  }
  __syncthreads();
  for (uint32_t item = blockIdx.x; item < count; item += gridDim.x) {
    const int s = __ldcg(P.near_list + item) - 1;
    if (s < 0 || s >= P.nseq) continue;
    const PassSeq ps = reinterpret_cast<const PassSeq *>(P.pseqw)[s];
    if (ps.j < 0 || ps.j > P.gamma) continue;  // not a drawn position: never use it as a row
    const TE *gp, *gq;
    draw_rows<TE>(P, s, ps.j, gp, gq);
    const bool vec =
        ((reinterpret_cast<uintptr_t>(gp) | reinterpret_cast<uintptr_t>(gq)) & 15u) == 0;
    const HpRow rp = hp_row(ps.dp, __ldg(P.Tp + s));
    const HpRow rq = ps.residual ? hp_row(ps.dq, __ldg(P.Tq + s)) : rp;
    psearch<TE>(P, ctl, s, ps, gp, gq, rp, rq, vec);
  }
}

// Slices of the draw and jobs of the precise redraw: slices of 16 steps
// (4096 entries) and about 64 precise jobs per draw, whole 256-entry steps
// each.
void set_chain_split(Params &P) {
  const int steps = P.steps;
  P.wj_steps = steps < 16 ? steps : 16;
  P.wj = (steps + P.wj_steps - 1) / P.wj_steps;
  const int kp = steps < 64 ? steps : 64;
  P.pj_steps = (steps + kp - 1) / kp;
  P.pj = (steps + P.pj_steps - 1) / P.pj_steps;
}

// Resident CTAs per SM of a kernel (cached per device and shared-memory size
// under a lock shared by every host thread).
struct OccCache {
  std::mutex mu;
  int dev = -1, smem = -1, blocks = 0;
};

template <typename K>
cudaError_t occupancy(OccCache &c, K kern, int threads, size_t smem, int &blocks) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(c.mu);
  if (dev != c.dev || static_cast<int>(smem) != c.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, threads, smem);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    c.blocks = per_sm * sms;
    c.dev = dev;
    c.smem = static_cast<int>(smem);
  }
  blocks = c.blocks;
  return cudaSuccess;
}

// Launch with programmatic stream serialisation: the kernel may begin while
// the previous one in the stream drains (it waits in grid_dependency_wait).
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

// Events a benchmark asked to be recorded around the rows kernel (both set
// or both null; see spec_set_profile_events).
std::mutex g_prof_mu;
cudaEvent_t g_prof_start = nullptr, g_prof_stop = nullptr;

template <typename TE>
cudaError_t launch_chain_t(Params P, const Exp2Table &tab, size_t smem, cudaStream_t stream) {
  cudaEvent_t prof_start, prof_stop;
  {
    std::lock_guard<std::mutex> lock(g_prof_mu);
    prof_start = g_prof_start;
    prof_stop = g_prof_stop;
  }
  static OccCache w_occ;
  int w_blocks = 0;
  cudaError_t e;
  set_chain_split(P);
  if (prof_start) {
    e = cudaEventRecord(prof_start, stream);
    if (e != cudaSuccess) return e;
  }
  e = launch_chain_rows(P, sizeof(TE), smem, stream);
  if (e != cudaSuccess) return e;
  if (prof_stop) {
    e = cudaEventRecord(prof_stop, stream);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(chain_decide_kernel<TE>, dim3(P.nseq), dim3(kKThreads), 0, stream, P);
  if (e != cudaSuccess) return e;
  // weights kernel: a ring of kWRing slots, each one slice of the p row and one
  // of the q row
  Params W = P;
  W.slot_bytes = static_cast<int>(static_cast<size_t>(P.wj_steps) * kStep * sizeof(TE));
  W.data_off = static_cast<int>((sizeof(WCtl) + 127) / 128 * 128);
  const size_t wsmem = W.data_off + static_cast<size_t>(kWRing) * 2 * W.slot_bytes;
  e = occupancy(w_occ, chain_weights_kernel<TE>, kWThreads, wsmem, w_blocks);
  if (e != cudaSuccess) return e;
  const long long witems = static_cast<long long>(P.nseq) * P.wj;
  e = launch_pdl(chain_weights_kernel<TE>, dim3(static_cast<int>(witems < w_blocks ? witems : w_blocks)),
                 dim3(kWThreads), wsmem, stream, W);
  if (e != cudaSuccess) return e;
  e = launch_pdl(chain_search_kernel<TE>, dim3(P.nseq), dim3(kDThreads), 0, stream, P);
  if (e != cudaSuccess) return e;
  const int gy = P.nseq < 32 ? P.nseq : 32;
  e = launch_pdl(chain_precise_kernel<TE>, dim3(P.pj, gy), dim3(kQThreads), 0, stream, P, tab);
  if (e != cudaSuccess) return e;
  return launch_pdl(chain_psearch_kernel<TE>, dim3(gy), dim3(kQThreads), 0, stream, P, tab);
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

}  // namespace sv
