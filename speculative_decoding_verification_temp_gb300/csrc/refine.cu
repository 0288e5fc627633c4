// Precise redraw of final draws that fell near a CDF boundary.
//
// The verification kernels draw in single precision: the token is the first
// index whose running weight sum exceeds u * Z.  Rounding in the exponentials,
// the normalisers and the running sums moves every boundary of that inverse
// CDF by up to a few 1e-7 of the probability mass, so when u * Z lands that
// close to a boundary the single-precision token can differ from the exact
// one.  Those draws are flagged (UnitOut::near) and queued by the path
// stitching; this kernel recomputes each queued draw with double-float weights
// (relative error below 1e-11) and double-precision sums, and overwrites the
// token.
//
// One thread-block cluster of 16 CTAs per queued draw, in a loop over the
// queue.  For a residual [p - c q]_+ the passes over the row pair are:
//   1. S_p, S_q: the softmax normalisers;
//   2. for a tree node whose held residual came after n > 1 rejections, the
//      multipliers c_1 = 1, c_{s+1} = c_s + W_s with W_s the total of
//      [p - c_s q]_+ (one pass each);
//   3. the weights of the final distribution, per-warp and per-CTA totals;
// then the inverse-CDF search: CTA, warp, then one warp scans its range.
// A draw from p itself needs only pass 3.  Rows are read from global memory
// in groups of 8 entries (16-byte loads when the rows are aligned): this path
// runs for a few percent of the draws.
#include <cooperative_groups.h>

#include "ops.cuh"
#include "precise.cuh"
#include "verify_units.cuh"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kRefineCluster = 16;

struct HpRow {
  float m;         // row maximum
  float khi, klo;  // log2(e) / T as a double-float
  float thr;       // top-k threshold (-inf: none)
};

__device__ __forceinline__ HpRow hp_row(const RowDesc &d, float T) {
  HpRow r;
  r.m = d.m;
  const Df k = df_from_double(1.44269504088896340735992468100189 / static_cast<double>(T));
  r.khi = k.hi;
  r.klo = k.lo;
  r.thr = d.thr;
  return r;
}

// exp((z - max) / T) as a double-float; 0 below the top-k threshold.
__device__ __forceinline__ Df hp_exp(const HpRow &r, float z, const float *th, const float *tl) {
  if (!(z > -INFINITY) || z < r.thr) return Df{0.f, 0.f};
  float dh, dl;
  two_sum(z, -r.m, dh, dl);  // z - max exactly
  const float t_hi = __fmul_rn(dh, r.khi);
  const float t_lo =
      __fadd_rn(fmaf(dh, r.khi, -t_hi), fmaf(dh, r.klo, __fmul_rn(dl, r.khi)));
  return df_exp2(df_norm(t_hi, t_lo), th, tl);
}

struct RefineSmem {
  float tab_hi[64], tab_lo[64];
  double wsum[2][kWarps];
  int wlast[kWarps];
  double cta[2];   // this CTA's totals, read by the cluster
  int cta_last;    // this CTA's last positive index (-1: none)
  int count;
  int token;
};

// Sum of (a, b) over the cluster; every thread gets the same values.
__device__ void cluster_sum2(double a, double b, double &A, double &B, RefineSmem &sm,
                             cg::cluster_group &cl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xFFFFFFFFu, a, off);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, off);
  }
  if (lane == 0) {
    sm.wsum[0][warp] = a;
    sm.wsum[1][warp] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    double ta = 0.0, tb = 0.0;
    for (int w = 0; w < kWarps; ++w) {
      ta += sm.wsum[0][w];
      tb += sm.wsum[1][w];
    }
    sm.cta[0] = ta;
    sm.cta[1] = tb;
  }
  cl.sync();
  A = 0.0;
  B = 0.0;
  for (int r = 0; r < kRefineCluster; ++r) {
    const double *x = cl.map_shared_rank(sm.cta, r);
    A += x[0];
    B += x[1];
  }
  cl.sync();
}

template <typename TE>
struct RefineRows {
  const TE *gp, *gq;
  HpRow rp, rq;
  int residual;
  int vec;  // both rows start on 16-byte boundaries
  Df rho;   // c S_p / S_q: the weight is [e_p - rho e_q]_+
};

// Logits of the 8 entries from `base` (a multiple of 8); -inf at or past `end`.
template <typename TE>
__device__ __forceinline__ void load8z(const TE *g, int base, int end, bool vec, float z[8]) {
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

// Weights of the 8 entries from `base` (0 at or past `end`).
template <typename TE>
__device__ __forceinline__ void hp_weight8(const RefineRows<TE> &R, int base, int end,
                                           const RefineSmem &sm, Df w[8]) {
  float zp[8], zq[8];
  load8z<TE>(R.gp, base, end, R.vec, zp);
  if (R.residual) load8z<TE>(R.gq, base, end, R.vec, zq);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const Df ep = hp_exp(R.rp, zp[e], sm.tab_hi, sm.tab_lo);
    if (!R.residual || ep.hi == 0.f) {
      w[e] = ep;
      continue;
    }
    const Df eq = hp_exp(R.rq, zq[e], sm.tab_hi, sm.tab_lo);
    const Df d = df_sub(ep, df_mul(R.rho, eq));
    w[e] = d.hi > 0.f ? d : Df{0.f, 0.f};
  }
}

// Sum of the 8 weights from `base` (entries at or past `end` are 0).
template <typename TE>
__device__ __forceinline__ double step_sum(const RefineRows<TE> &R, int base, int end,
                                           const RefineSmem &sm, int &lastpos) {
  Df w[8];
  hp_weight8(R, base, end, sm, w);
  Df s{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (w[e].hi > 0.f) lastpos = base + e;
    s = df_add(s, w[e]);
  }
  return df_to_double(s);
}

template <typename TE>
__global__ void __cluster_dims__(kRefineCluster, 1, 1) __launch_bounds__(kThreads)
    refine_kernel(const Params P, const Exp2Table tab) {
  __shared__ RefineSmem sm;
  cg::cluster_group cl = cg::this_cluster();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int rank = static_cast<int>(cl.block_rank());
  const int cid = blockIdx.x / kRefineCluster, G = gridDim.x / kRefineCluster;
  for (int i = tid; i < 64; i += kThreads) {
    sm.tab_hi[i] = tab.hi[i];
    sm.tab_lo[i] = tab.lo[i];
  }
  if (tid == 0) sm.count = min(static_cast<int>(*reinterpret_cast<volatile uint32_t *>(P.refine_ctr)),
                              P.nseq);
  __syncthreads();
  const int count = sm.count;
  const int V = P.V;
  // this CTA's range, and each warp's contiguous part of it
  const int Ls = ((V + kRefineCluster - 1) / kRefineCluster + 7) / 8 * 8;
  const int v0 = min(V, rank * Ls), v1 = min(V, v0 + Ls);
  const int Lw = ((Ls + kWarps - 1) / kWarps + 255) / 256 * 256;
  const int ws = min(v1, v0 + warp * Lw), we = min(v1, ws + Lw);

  for (int item = cid; item < count; item += G) {
    const int4 it = P.refine[item];
    const int seq = it.x, unit = it.y, pos = it.z;
    const UnitStats st = P.stats[unit];
    const int node = st.node;
    long long prow, qrow;
    if (P.mode == kModeChain) {
      prow = static_cast<long long>(seq) * (P.gamma + 1) + node;
      qrow = static_cast<long long>(seq) * P.gamma + node;
    } else {
      prow = qrow = static_cast<long long>(seq) * P.ups + node;
    }
    RefineRows<TE> R;
    R.gp = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE)));
    R.gq = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE)));
    R.rp = hp_row(st.p, __ldg(P.Tp + seq));
    R.residual = st.c > 0.f && st.n_res > 0;
    R.vec = ((reinterpret_cast<uintptr_t>(R.gp) | reinterpret_cast<uintptr_t>(R.gq)) & 15u) == 0;
    R.rho = Df{0.f, 0.f};
    if (R.residual) {
      R.rq = hp_row(st.q, __ldg(P.Tq + seq));
      // pass 1: the normalisers
      Df sp{0.f, 0.f}, sq{0.f, 0.f};
      for (int base = ws + lane * 8; base < we; base += 256) {
        float zp[8], zq[8];
        load8z<TE>(R.gp, base, we, R.vec, zp);
        load8z<TE>(R.gq, base, we, R.vec, zq);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sp = df_add(sp, hp_exp(R.rp, zp[e], sm.tab_hi, sm.tab_lo));
          sq = df_add(sq, hp_exp(R.rq, zq[e], sm.tab_hi, sm.tab_lo));
        }
      }
      double Sp, Sq;
      cluster_sum2(df_to_double(sp), df_to_double(sq), Sp, Sq, sm, cl);
      // pass 2: the multiplier of the held residual
      double c = 1.0;
      for (int s = 1; s < st.n_res; ++s) {
        R.rho = df_from_double(c * Sp / Sq);
        double part = 0.0;
        int lp = -1;
        for (int base = ws + lane * 8; base < we; base += 256) part += step_sum(R, base, we, sm, lp);
        double W, unused;
        cluster_sum2(part, 0.0, W, unused, sm, cl);
        c += W / Sp;
      }
      R.rho = df_from_double(c * Sp / Sq);
    }
    // pass 3: weights of the final distribution, per-warp and per-CTA totals
    double part = 0.0;
    int lp = -1;
    for (int base = ws + lane * 8; base < we; base += 256) part += step_sum(R, base, we, sm, lp);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
      lp = max(lp, __shfl_xor_sync(0xFFFFFFFFu, lp, off));
    }
    if (lane == 0) {
      sm.wsum[0][warp] = part;
      sm.wlast[warp] = lp;
    }
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      int l = -1;
      for (int w = 0; w < kWarps; ++w) {
        t += sm.wsum[0][w];
        l = max(l, sm.wlast[w]);
      }
      sm.cta[0] = t;
      sm.cta_last = l;
    }
    cl.sync();
    // the owning CTA: the same prefix in every CTA
    const double u = static_cast<double>(unit_uniform(P, seq, node, 1));
    double Z = 0.0;
    double totals[kRefineCluster];
    int lasts[kRefineCluster];
    for (int r = 0; r < kRefineCluster; ++r) {
      RefineSmem *o = cl.map_shared_rank(&sm, r);
      totals[r] = o->cta[0];
      lasts[r] = o->cta_last;
      Z += totals[r];
    }
    const double t = u * Z;
    int owner = -1;
    double trel = 0.0;
    {
      double acc = 0.0;
      for (int r = 0; r < kRefineCluster; ++r) {
        if (acc + totals[r] > t) {
          owner = r;
          trel = t - acc;
          break;
        }
        acc += totals[r];
      }
    }
    bool fallback = false;
    if (owner < 0) {
      fallback = true;
      for (int r = kRefineCluster - 1; r >= 0; --r)
        if (lasts[r] >= 0) {
          owner = r;
          break;
        }
    }
    cl.sync();  // every DSMEM read of this item is done
    if (rank == owner) {
      if (tid == 0) {
        int tok = sm.cta_last;
        int ow = -1;
        double wt = 0.0;
        if (!fallback) {
          double acc = 0.0;
          for (int w = 0; w < kWarps; ++w) {
            if (acc + sm.wsum[0][w] > trel) {
              ow = w;
              wt = trel - acc;
              break;
            }
            acc += sm.wsum[0][w];
          }
        }
        sm.token = ow < 0 ? tok : -1 - ow;  // >= 0: decided; else the warp to scan
        sm.wsum[1][0] = wt;
      }
      __syncthreads();
      const int code = sm.token;
      if (code < 0 && warp == -1 - code) {
        const double wt = sm.wsum[1][0];
        double base_sum = 0.0;
        int result = -1;
        for (int rb = ws; rb < we && result < 0; rb += 256) {
          const int base = rb + lane * 8;
          Df wd[8];
          hp_weight8(R, base, we, sm, wd);
          double w[8];
          double s = 0.0;
          int lpos = -1;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            w[e] = df_to_double(wd[e]);
            s += w[e];
            if (w[e] > 0.0) lpos = base + e;
          }
          double incl = s;
#pragma unroll
          for (int off = 1; off < 32; off <<= 1) {
            const double x = __shfl_up_sync(0xFFFFFFFFu, incl, off);
            if (lane >= off) incl += x;
          }
          double excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
          if (lane == 0) excl = 0.0;
          const unsigned hit = __ballot_sync(0xFFFFFFFFu, base_sum + incl > wt);
          if (hit) {
            const int first = __ffs(hit) - 1;
            int found = -1;
            if (lane == first) {
              double run = base_sum + excl;
#pragma unroll
              for (int e = 0; e < 8; ++e) {
                run += w[e];
                if (found < 0 && w[e] > 0.0 && run > wt) found = base + e;
              }
              if (found < 0) found = lpos;
            }
            result = __shfl_sync(0xFFFFFFFFu, found, first);
          }
          base_sum += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
        if (lane == 0) sm.token = result >= 0 ? result : sm.wlast[warp];
      }
      __syncthreads();
      if (tid == 0 && sm.token >= 0) {
        const int width = P.mode == kModeChain ? P.gamma + 1 : P.max_depth + 1;
        P.outs[unit].token = sm.token;
        P.out_tokens[static_cast<long long>(seq) * width + pos] = sm.token;
      }
    }
    __syncthreads();
  }
}

template <typename TE>
cudaError_t launch_refine_t(const Params &P, const Exp2Table &tab, cudaStream_t stream) {
  static bool attr_set = false;  // clusters of 16 need the non-portable size opt-in
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(
        refine_kernel<TE>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  const int G = P.nseq < 9 ? P.nseq : 9;  // 144 CTAs: one wave on 152 SMs
  refine_kernel<TE><<<dim3(G * kRefineCluster), kThreads, 0, stream>>>(P, tab);
  return cudaGetLastError();
}

cudaError_t launch_refine(const Params &P, int esize, const Exp2Table &tab, cudaStream_t stream) {
  return esize == 2 ? launch_refine_t<uint16_t>(P, tab, stream)
                    : launch_refine_t<float>(P, tab, stream);
}

}  // namespace sv
