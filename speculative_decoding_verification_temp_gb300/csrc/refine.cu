// Precise redraw of final draws that fell near a CDF boundary.
//
// The verification kernels draw in single precision: the token is the first
// index whose running weight sum exceeds u * Z.  Rounding in the exponentials,
// the normalisers and the running sums moves every boundary of that inverse
// CDF by up to a few 1e-7 of the probability mass, so when u * Z lands that
// close to a boundary the single-precision token can differ from the exact
// one.  Those draws are flagged (UnitOut::near) and queued; this kernel
// recomputes each queued draw with double-float weights (relative error below
// 1e-11) and double-precision sums, and overwrites the token.
//
// The whole grid works on the queue at once: with `count` queued draws and G
// CTAs, each draw's vocabulary is cut into S = max(1, G / count) slices and
// work unit u (draw u / S, slice u % S) goes to CTA u mod G.  Phases are
// separated by a grid barrier (the launch is cooperative, so every CTA is
// resident; each wait is bounded):
//   A. for a residual [p - c q]_+: each unit's share of the softmax
//      normalisers S_p, S_q;
//   R. for a tree node whose held residual came after n > 1 rejections, the
//      multipliers c_1 = 1, c_{s+1} = c_s + W_s / S_p with W_s the total of
//      [e_p - c_s (S_p / S_q) e_q]_+ (two barriers per round);
//   B. the final weights: per-warp totals and last positive entries of each
//      unit, published in the workspace;
//   C. every unit sums its draw's slice totals in the same fixed order (so all
//      of them see the same Z), finds the owning slice and, if it owns it,
//      the owning warp, which scans its range with a warp prefix sum.
// A draw from p itself needs only B and C.  Rows are read from global memory
// in groups of 8 entries (16-byte loads when the rows are aligned).
#include <mutex>

#include "ops.cuh"
#include "precise_row.cuh"

namespace sv {

constexpr long long kRefineWaitNs = 2000000000ll;  // give up a barrier after about 2 s

struct RefineSmem {
  float tab_hi[64], tab_lo[64];
  double red[2][kWarps];
  int redi[kWarps];
  int count;
  int nres_max;
  int any_residual;
  int abort;
  int token;
  int owner_warp;
  double wt;
};

// One queued draw and the rows it is taken from.
template <typename TE>
struct RefineItem {
  int seq, unit, pos;
  int node;      // the node drawn at (its id keys the draw uniform)
  int residual;  // weights [e_p - rho e_q]_+ (else e_p)
  int n_res;
  const TE *gp, *gq;
  HpRow rp, rq;
  int vec;       // both rows start on 16-byte boundaries
};

template <typename TE>
__device__ RefineItem<TE> load_item(const Params &P, int item) {
  const int4 q = P.refine[item];
  RefineItem<TE> it;
  it.seq = q.x;
  it.unit = q.y;
  it.pos = q.z;
  const UnitStats st = P.stats[it.unit];
  const int node = st.node;
  it.node = node;
  long long prow, qrow;
  if (P.mode == kModeChain) {
    prow = static_cast<long long>(it.seq) * (P.gamma + 1) + node;
    qrow = static_cast<long long>(it.seq) * P.gamma + node;
  } else {
    prow = qrow = static_cast<long long>(it.seq) * P.ups + node;
  }
  it.gp = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE)));
  it.gq = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE)));
  it.rp = hp_row(st.p, __ldg(P.Tp + it.seq));
  it.residual = st.c > 0.f && st.n_res > 0;
  it.n_res = it.residual ? st.n_res : 0;
  it.rq = it.residual ? hp_row(st.q, __ldg(P.Tq + it.seq)) : it.rp;
  it.vec = ((reinterpret_cast<uintptr_t>(it.gp) | reinterpret_cast<uintptr_t>(it.gq)) & 15u) == 0;
  return it;
}

// Weights of the 8 entries from `base` (0 at or past `end`); rho = c S_p / S_q.
template <typename TE>
__device__ __forceinline__ void hp_weight8(const RefineItem<TE> &it, Df rho, int base, int end,
                                           const RefineSmem &sm, Df w[8]) {
  float zp[8], zq[8];
  hp_load8<TE>(it.gp, base, end, it.vec, zp);
  if (it.residual) hp_load8<TE>(it.gq, base, end, it.vec, zq);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const Df ep = hp_exp(it.rp, zp[e], sm.tab_hi, sm.tab_lo);
    if (!it.residual || ep.hi == 0.f) {
      w[e] = ep;
      continue;
    }
    const Df eq = hp_exp(it.rq, zq[e], sm.tab_hi, sm.tab_lo);
    const Df d = df_sub(ep, df_mul(rho, eq));
    w[e] = d.hi > 0.f ? d : Df{0.f, 0.f};
  }
}

// Sum of the 8 weights from `base`; `lastpos` becomes the last positive entry.
template <typename TE>
__device__ __forceinline__ double step_sum(const RefineItem<TE> &it, Df rho, int base, int end,
                                           const RefineSmem &sm, int &lastpos) {
  Df w[8];
  hp_weight8(it, rho, base, end, sm, w);
  Df s{0.f, 0.f};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    if (w[e].hi > 0.f) lastpos = base + e;
    s = df_add(s, w[e]);
  }
  return df_to_double(s);
}

// Vocabulary range of slice k of S, and warp w's contiguous part of it (whole
// groups of 256 entries, so each lane's groups of 8 stay aligned).
struct SliceRange {
  int v0, v1, ws, we;
};

__device__ __forceinline__ SliceRange slice_range(int V, int S, int k, int warp) {
  SliceRange r;
  const int Ls = ((V + S - 1) / S + 7) / 8 * 8;
  r.v0 = min(V, k * Ls);
  r.v1 = min(V, r.v0 + Ls);
  const int Lw = ((Ls + kWarps - 1) / kWarps + 255) / 256 * 256;
  r.ws = min(r.v1, r.v0 + warp * Lw);
  r.we = min(r.v1, r.ws + Lw);
  return r;
}

// Sum over the block of two doubles (thread 0 gets the totals).
__device__ __forceinline__ void block_sum2(double &a, double &b, RefineSmem &sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    a += __shfl_xor_sync(0xFFFFFFFFu, a, off);
    b += __shfl_xor_sync(0xFFFFFFFFu, b, off);
  }
  if (lane == 0) {
    sm.red[0][warp] = a;
    sm.red[1][warp] = b;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    a = 0.0;
    b = 0.0;
    for (int w = 0; w < kWarps; ++w) {
      a += sm.red[0][w];
      b += sm.red[1][w];
    }
  }
  __syncthreads();
}

// Grid barrier number `idx` (0, 1, ...): every CTA adds one to the counter and
// waits until all G have added for this barrier.  Bounded: a wait that runs out
// sets error bit 1 and makes the CTA stop working on the queue.
__device__ bool grid_barrier(const Params &P, RefineSmem &sm, int idx) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(P.rbar) : "memory");
    const uint32_t target = static_cast<uint32_t>(gridDim.x) * static_cast<uint32_t>(idx + 1);
    long long t0;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
    int ok = 1;
    while (true) {
      uint32_t v;
      asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(P.rbar) : "memory");
      if (v >= target) break;
      long long t;
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
      if (t - t0 > kRefineWaitNs) {
        ok = 0;
        atomicOr(P.err, 2u);
        break;
      }
      __nanosleep(64);
    }
    sm.abort = ok ? 0 : 1;
  }
  __syncthreads();
  return sm.abort == 0;
}

// Sum over the S units of a draw of one field: lane-strided partial sums and a
// shuffle tree, then lane 0's value for every lane, so each warp of each CTA
// gets the same bits.
template <typename F>
__device__ __forceinline__ double units_sum(int S, F field) {
  const int lane = threadIdx.x & 31;
  double s = 0.0;
  for (int k = lane; k < S; k += 32) s += field(k);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xFFFFFFFFu, s, off);
  return __shfl_sync(0xFFFFFFFFu, s, 0);
}

// (S_p, S_q) of a draw: the sum of its units' phase-A partials.
__device__ __forceinline__ void item_normalisers(const Params &P, int item, int S, double &Sp,
                                                 double &Sq) {
  const RefinePart *x = P.rpart + static_cast<long long>(item) * S;
  Sp = units_sum(S, [&](int k) { return __ldcg(&x[k].a); });
  Sq = units_sum(S, [&](int k) { return __ldcg(&x[k].b); });
}

template <typename TE>
__global__ void __launch_bounds__(kThreads) refine_kernel(const Params P, const Exp2Table tab) {
  __shared__ RefineSmem sm;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  for (int i = tid; i < 64; i += kThreads) {
    sm.tab_hi[i] = tab.hi[i];
    sm.tab_lo[i] = tab.lo[i];
  }
  if (tid == 0) sm.count = min(static_cast<int>(*reinterpret_cast<volatile uint32_t *>(P.refine_ctr)),
                              P.nseq);
  __syncthreads();
  const int count = sm.count;
  if (count <= 0) return;  // the same decision in every CTA
  const int V = P.V;
  const int S = max(1, G / count);
  const int U = count * S;
  // the largest residual round count and whether any draw is a residual
  {
    int nr = 0, anyr = 0;
    for (int item = tid; item < count; item += kThreads) {
      const UnitStats st = P.stats[P.refine[item].y];
      if (st.c > 0.f && st.n_res > 0) {
        anyr = 1;
        nr = max(nr, st.n_res);
      }
    }
    nr = warp_max_i(nr);
    anyr = warp_max_i(anyr);
    if (lane == 0) {
      sm.redi[warp] = nr;
      sm.red[0][warp] = anyr;
    }
    __syncthreads();
    if (tid == 0) {
      int a = 0, b = 0;
      for (int w = 0; w < kWarps; ++w) {
        a = max(a, sm.redi[w]);
        b = max(b, static_cast<int>(sm.red[0][w]));
      }
      sm.nres_max = a;
      sm.any_residual = b;
    }
    __syncthreads();
  }
  const int nres_max = sm.nres_max;
  int bar = 0;
  // A: shares of the softmax normalisers of residual draws
  if (sm.any_residual) {
    for (int u = blockIdx.x; u < U; u += G) {
      const int item = u / S, k = u - item * S;
      const RefineItem<TE> it = load_item<TE>(P, item);
      if (!it.residual) continue;
      const SliceRange r = slice_range(V, S, k, warp);
      Df sp{0.f, 0.f}, sq{0.f, 0.f};
#pragma unroll 4
      for (int base = r.ws + lane * 8; base < r.we; base += 256) {
        float zp[8], zq[8];
        hp_load8<TE>(it.gp, base, r.we, it.vec, zp);
        hp_load8<TE>(it.gq, base, r.we, it.vec, zq);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          sp = df_add(sp, hp_exp(it.rp, zp[e], sm.tab_hi, sm.tab_lo));
          sq = df_add(sq, hp_exp(it.rq, zq[e], sm.tab_hi, sm.tab_lo));
        }
      }
      double a = df_to_double(sp), b = df_to_double(sq);
      block_sum2(a, b, sm);
      if (tid == 0) {
        P.rpart[u].a = a;
        P.rpart[u].b = b;
        if (k == 0) P.rc[item] = 1.0;
      }
    }
    if (!grid_barrier(P, sm, bar++)) return;
  }
  // R: multipliers of residuals held after several rejections (trees)
  for (int s = 1; s < nres_max; ++s) {
    for (int u = blockIdx.x; u < U; u += G) {
      const int item = u / S, k = u - item * S;
      const RefineItem<TE> it = load_item<TE>(P, item);
      if (!it.residual || s >= it.n_res) continue;
      double Sp, Sq;
      item_normalisers(P, item, S, Sp, Sq);
      const Df rho = df_from_double(__ldcg(P.rc + item) * Sp / Sq);
      const SliceRange r = slice_range(V, S, k, warp);
      double part = 0.0, unused = 0.0;
      int lp = -1;
#pragma unroll 4
      for (int base = r.ws + lane * 8; base < r.we; base += 256)
        part += step_sum(it, rho, base, r.we, sm, lp);
      block_sum2(part, unused, sm);
      if (tid == 0) P.rpart[u].rw = part;
    }
    if (!grid_barrier(P, sm, bar++)) return;
    for (int item = blockIdx.x; item < count && warp == 0; item += G) {
      const UnitStats st = P.stats[P.refine[item].y];
      if (!(st.c > 0.f && st.n_res > 0) || s >= st.n_res) continue;
      double Sp, Sq;
      item_normalisers(P, item, S, Sp, Sq);
      const RefinePart *x = P.rpart + static_cast<long long>(item) * S;
      const double W = units_sum(S, [&](int k) { return __ldcg(&x[k].rw); });
      if (lane == 0) P.rc[item] = __ldcg(P.rc + item) + W / Sp;
    }
    if (!grid_barrier(P, sm, bar++)) return;
  }
  // B: final weights, per-warp totals of each unit
  for (int u = blockIdx.x; u < U; u += G) {
    const int item = u / S, k = u - item * S;
    const RefineItem<TE> it = load_item<TE>(P, item);
    Df rho{0.f, 0.f};
    if (it.residual) {
      double Sp, Sq;
      item_normalisers(P, item, S, Sp, Sq);
      rho = df_from_double(__ldcg(P.rc + item) * Sp / Sq);
    }
    const SliceRange r = slice_range(V, S, k, warp);
    double part = 0.0;
    int lp = -1;
#pragma unroll 4
    for (int base = r.ws + lane * 8; base < r.we; base += 256)
      part += step_sum(it, rho, base, r.we, sm, lp);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      part += __shfl_xor_sync(0xFFFFFFFFu, part, off);
      lp = max(lp, __shfl_xor_sync(0xFFFFFFFFu, lp, off));
    }
    if (lane == 0) {
      P.rpart[u].warp[warp] = part;
      P.rpart[u].wlast[warp] = lp;
      sm.red[0][warp] = part;
      sm.redi[warp] = lp;
    }
    __syncthreads();
    if (tid == 0) {
      double t = 0.0;
      int l = -1;
      for (int w = 0; w < kWarps; ++w) {
        t += sm.red[0][w];
        l = max(l, sm.redi[w]);
      }
      P.rpart[u].w = t;
      P.rpart[u].last = l;
    }
    __syncthreads();
  }
  if (!grid_barrier(P, sm, bar++)) return;
  // C: the owning slice, warp and entry
  for (int u = blockIdx.x; u < U; u += G) {
    const int item = u / S, k = u - item * S;
    const RefineItem<TE> it = load_item<TE>(P, item);
    if (warp == 0) {
      // the owning slice: lanes hold contiguous runs of slices, a warp scan
      // of the run totals finds the lane, that lane walks its run
      const RefinePart *parts = P.rpart + static_cast<long long>(item) * S;
      const int per = (S + 31) / 32;
      const int s0 = min(S, lane * per), s1 = min(S, s0 + per);
      double seg = 0.0;
      int lastslice = -1;
      for (int x = s0; x < s1; ++x) {
        seg += __ldcg(&parts[x].w);
        if (__ldcg(&parts[x].last) >= 0) lastslice = x;
      }
      double incl = seg;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += y;
      }
      const double Z = __shfl_sync(0xFFFFFFFFu, incl, 31);
      const double t = static_cast<double>(unit_uniform(P, it.seq, it.node, 1)) * Z;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > t && seg > 0.0);
      int owner = -1;
      double trel = 0.0;
      if (hit) {
        const int first = __ffs(hit) - 1;
        if (lane == first) {
          double acc = incl - seg;
          for (int x = s0; x < s1; ++x) {
            const double tx = __ldcg(&parts[x].w);
            if (acc + tx > t && tx > 0.0) {
              owner = x;
              trel = t - acc;
              break;
            }
            acc += tx;
          }
        }
        owner = __shfl_sync(0xFFFFFFFFu, owner, first);
        trel = __shfl_sync(0xFFFFFFFFu, trel, first);
      }
      int token = -2;  // -2: not this unit's; -1: scan warp sm.owner_warp
      if (owner < 0) {
        // rounding left no entry above u * Z: the last slice with a positive entry
        const int fb = warp_max_i(lastslice);
        if (fb == k) token = __ldcg(&parts[k].last);
      } else if (owner == k) {
        // the owning warp: a scan of the unit's eight warp totals
        const double x = lane < kWarps ? __ldcg(&parts[k].warp[lane]) : 0.0;
        double wi = x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const double y = __shfl_up_sync(0xFFFFFFFFu, wi, off);
          if (lane >= off) wi += y;
        }
        const unsigned wh = __ballot_sync(0xFFFFFFFFu, lane < kWarps && wi > trel);
        if (wh) {
          const int ow = __ffs(wh) - 1;
          const double wt = trel - __shfl_sync(0xFFFFFFFFu, wi - x, ow);
          token = -1;
          if (lane == 0) {
            sm.owner_warp = ow;
            sm.wt = wt;
          }
        } else {
          token = __ldcg(&parts[k].last);
        }
      }
      if (lane == 0) sm.token = token;
    }
    __syncthreads();
    if (sm.token == -1 && warp == sm.owner_warp) {
      const double wt = sm.wt;
      const SliceRange r = slice_range(V, S, k, warp);
      Df rho{0.f, 0.f};
      if (it.residual) {
        double Sp, Sq;
        item_normalisers(P, item, S, Sp, Sq);
        rho = df_from_double(__ldcg(P.rc + item) * Sp / Sq);
      }
      double base_sum = 0.0;
      int result = -1;
      for (int rb = r.ws; rb < r.we && result < 0; rb += 256) {
        const int base = rb + lane * 8;
        Df wd[8];
        hp_weight8(it, rho, base, r.we, sm, wd);
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
      if (lane == 0)
        sm.token = result >= 0 ? result : __ldcg(&P.rpart[u].wlast[warp]);
    }
    __syncthreads();
    if (tid == 0 && sm.token >= 0) {
      const int width = P.mode == kModeChain ? P.gamma + 1 : P.max_depth + 1;
      P.outs[it.unit].token = sm.token;
      P.out_tokens[static_cast<long long>(it.seq) * width + it.pos] = sm.token;
    }
    __syncthreads();
  }
}

template <typename TE>
cudaError_t launch_refine_t(const Params &P, const Exp2Table &tab, cudaStream_t stream) {
  static std::mutex mu;  // guards the cache below across host threads
  static int cached_dev = -1, cached_blocks = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::unique_lock<std::mutex> lock(mu);
  if (dev != cached_dev) {
    int per_sm = 0, sms = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, refine_kernel<TE>, kThreads, 0);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    cached_blocks = min(kRefineMaxGrid, min(per_sm, 2) * sms);
    cached_dev = dev;
  }
  const int blocks = cached_blocks;
  lock.unlock();
  void *args[] = {const_cast<Params *>(&P), const_cast<Exp2Table *>(&tab)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(refine_kernel<TE>),
                                     dim3(blocks), dim3(kThreads), args, 0, stream);
}

cudaError_t launch_refine(const Params &P, int esize, const Exp2Table &tab, cudaStream_t stream) {
  return esize == 2 ? launch_refine_t<uint16_t>(P, tab, stream)
                    : launch_refine_t<float>(P, tab, stream);
}

}  // namespace sv
