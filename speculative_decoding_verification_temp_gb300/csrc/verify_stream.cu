// Streaming verification kernel: a cooperative persistent grid of
// independent CTAs fed by a task scheduler in each CTA.
//
// A unit's target (+ draft) row is cut into C slices of at most 32 KB.  Two
// kinds of task exist:
//   stats   (u, r): online max / sum (argmax for temperature 0) of slice r of
//                   unit u's rows; every unit has C of them, handed out
//                   statically (CTA b takes tasks b, b + gridDim, ... in
//                   unit-major order, so the slices of a unit stream together);
//   weights (u, r, round): the draw weights of slice r - [p - c q]_+ after a
//                   rejection, or p for a bonus draw - summed per block of
//                   about 500 entries; created on demand and taken by
//                   whichever CTA claims them first from a global queue.
// Each CTA has a producer warp whose lane 0 is the scheduler: it claims a
// queued weight task if there is one, else its next stats task, and streams
// the task's chunks (at most 16 KB each) through a four-slot shared-memory
// ring with bulk asynchronous copies (cp.async.bulk; a "full" and an "empty"
// mbarrier per slot).  The 256 compute threads process whatever arrives and
// hand each slot straight back.  A task's result goes to the workspace and
// bumps a per-unit counter; the CTA that completes a unit's stats merges the
// slices and tests the node's children; when it must draw it queues the C
// weight tasks, and the CTA that completes a weight round finishes it: the
// next child's test (trees), another round, or the inverse-CDF draw (owning
// block from the block totals, then one warp scans that block).  Weight tasks
// re-read slices streamed a few microseconds earlier, so they hit L2 and HBM
// sees every logit byte once.  No CTA waits on another except the schedulers'
// bounded polling of the queue once their stats tasks are done, which is why
// the grid is launched cooperatively (all CTAs resident).  A second small
// kernel stitches each sequence's path.
#include <mutex>

#include "ops.cuh"

namespace sv {

constexpr int kProducerWarp = kWarps;         // warp 8
constexpr int kBlockThreads = kThreads + 32;  // 256 compute threads + the producer warp
constexpr long long kPollLimitNs = 2000000000ll;  // give up polling after about 2 s

struct UnitInfo {
  int seq, node;
  long long prow, qrow;
  int p_arg, q_arg, tp_bad, tq_bad, load_q, has_children;
  float kp, kq;
};

__device__ __forceinline__ UnitInfo decode_unit(const Params &P, int unit) {
  UnitInfo u;
  u.seq = unit / P.ups;
  u.node = unit % P.ups;
  const float Tp = __ldg(P.Tp + u.seq), Tq = __ldg(P.Tq + u.seq);
  u.tp_bad = !(Tp >= 0.f) || Tp == INFINITY;
  u.tq_bad = !(Tq >= 0.f) || Tq == INFINITY;
  u.p_arg = u.tp_bad || Tp == 0.f;
  u.q_arg = u.tq_bad || Tq == 0.f;
  u.kp = u.p_arg ? 0.f : kLog2e / Tp;
  u.kq = u.q_arg ? 0.f : kLog2e / Tq;
  if (P.mode == kModeChain) {
    u.prow = static_cast<long long>(u.seq) * (P.gamma + 1) + u.node;
    u.qrow = static_cast<long long>(u.seq) * P.gamma + u.node;
    u.has_children = u.node < P.gamma;
  } else {
    u.prow = static_cast<long long>(u.seq) * P.ups + u.node;
    u.qrow = u.prow;
    u.has_children = __ldg(P.first_child + unit) >= 0;
  }
  u.load_q = u.has_children && !u.p_arg;
  return u;
}

__device__ __forceinline__ void mbar_arrive(unsigned long long *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint32_t ld_volatile(const uint32_t *p) {
  return *reinterpret_cast<const volatile uint32_t *>(p);
}

__device__ __forceinline__ long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return static_cast<long long>(t);
}

// A unit's draw state, read through L2 (another SM may have written it since
// this SM last looked).
__device__ __forceinline__ DrawState load_dstate(const DrawState *src) {
  DrawState d;
  const int4 *s4 = reinterpret_cast<const int4 *>(src);
  int4 *d4 = reinterpret_cast<int4 *>(&d);
#pragma unroll
  for (int i = 0; i < static_cast<int>(sizeof(DrawState) / 16); ++i) d4[i] = __ldcg(s4 + i);
  return d;
}

// Slice geometry of slice r.
struct SliceGeo {
  int v0, len, nvec;
};
__device__ __forceinline__ SliceGeo slice_geo(const Params &P, int r, int esize) {
  SliceGeo s;
  s.v0 = r * P.slice;
  s.len = max(0, min(P.V, s.v0 + P.slice) - s.v0);
  s.nvec = (s.len * esize) / 16;
  return s;
}

// Element range [bs, be) (vocabulary indices) of draw block b of slice r.
__device__ __forceinline__ void block_range(const Params &P, int r, int b, int esize, int &bs,
                                            int &be) {
  const SliceGeo g = slice_geo(P, r, esize);
  const int pe = 16 / esize;
  const int cvec = P.slot_bytes / 16;
  const int ce = cvec * pe;
  const int bl = ((ce + kBlocksPerChunk - 1) / kBlocksPerChunk + 7) / 8 * 8;
  const int nchunk_blocks = P.chunks * kBlocksPerChunk;
  if (b == nchunk_blocks) {  // the ragged tail
    bs = g.v0 + g.nvec * pe;
    be = g.v0 + g.len;
    return;
  }
  const int cc = b / kBlocksPerChunk, bi = b % kBlocksPerChunk;
  const int cn = max(0, min(cvec, g.nvec - cc * cvec)) * pe;  // entries in the chunk
  const int s = min(cn, bi * bl), e = min(cn, s + bl);
  bs = g.v0 + cc * ce + s;
  be = g.v0 + cc * ce + e;
}

// ---------------------------------------------------------------------------
// unit outcome
// ---------------------------------------------------------------------------

__device__ void publish_unit(const Params &P, int unit, int node, int next, int token,
                             uint32_t flags, const RowDesc &dp, const RowDesc &dq, float c,
                             float total, int kind, int near = 0, int n_res = 0) {
  UnitOut o;
  o.next = next;
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
  st.node = node;
  st.n_res = n_res;
  st.pad = 0;
  P.stats[unit] = st;
  P.unit_done[unit] = 0u;  // leave the counters zeroed for the next call
  P.w_done[unit] = 0u;
  __threadfence();
  atomicAdd(P.wq_ctr + 2, 1u);
}

// Queue the C weight tasks of the next round of unit u (thread 0 only).
__device__ void enqueue_round(const Params &P, int unit, DrawState &ds) {
  const int C = P.cluster;
  ds.round += 1;
  P.dstate[unit] = ds;
  __threadfence();
  const uint32_t idx = atomicAdd(P.wq_ctr + 1, static_cast<uint32_t>(C));
  for (int r = 0; r < C; ++r) {
    if (static_cast<long long>(idx) + r >= P.wq_cap) break;  // sized on the host: never hit
    int4 *e = P.wq + idx + r;
    e->x = unit;
    e->y = r;
    e->z = ds.round;
  }
  __threadfence();
  for (int r = 0; r < C; ++r) {
    if (static_cast<long long>(idx) + r >= P.wq_cap) break;
    reinterpret_cast<volatile int *>(P.wq + idx + r)[3] = static_cast<int>(P.epoch);
  }
}

// Next child of `node` after `after` (single thread; trees scan the parents).
__device__ int next_child_1(const Params &P, int seq, int node, int after) {
  if (P.mode == kModeChain) return (node < P.gamma && after < node + 1) ? node + 1 : -1;
  const int32_t *par = P.parent + static_cast<long long>(seq) * P.ups;
  for (int c = max(after, node) + 1; c < P.ups; ++c)
    if (__ldg(par + c) == node) return c;
  return -1;
}

// Test the children of the node from `child` on with the held distribution
// (thread 0).  Returns the accepted child or -1; `child` is left at the last
// child tested (rejected) and `rejected` says whether one was.
template <typename TE>
__device__ int test_children(const Params &P, const UnitInfo &u, DrawState &ds, int &child,
                             bool stop_after_reject, bool &rejected) {
  const int V = P.V;
  const TE *gp = static_cast<const TE *>(row_ptr(P.target, u.prow, P.ld_t, sizeof(TE)));
  const TE *gq = static_cast<const TE *>(row_ptr(P.draft, u.qrow, P.ld_d, sizeof(TE)));
  rejected = false;
  while (child >= 0) {
    const int x = child_token(P, u.seq, u.node, child);
    const float uu = unit_uniform(P, u.seq, P.mode == kModeChain ? u.node : child, 0);
    int verdict = 0;
    if (x < 0 || x >= V) {
      ds.flags |= SPEC_FLAG_BAD_TOKEN;
    } else {
      const float zpx = to_f32(gp[x]);
      const float zqx = ds.dq.onehot ? 0.f : to_f32(gq[x]);
      const float qx = prob(ds.dq, zqx, x);
      if (!(qx > 0.f)) {
        ds.flags |= SPEC_FLAG_ZERO_Q;
      } else {
        const float px = ds.c_cur > 0.f ? weight(ds.dp, ds.dq, 1, ds.c_cur, zpx, zqx, x) / ds.W_cur
                                        : prob(ds.dp, zpx, x);
        verdict = uu < fminf(1.f, px / qx) ? 1 : 0;
      }
    }
    ds.child = child;
    if (verdict == 1) return child;
    rejected = true;
    if (stop_after_reject) return -1;
    child = next_child_1(P, u.seq, u.node, child);
  }
  return -1;
}

// Scan [bs, be) with one warp for the first running weight above t; on a
// rounding miss, the last positive entry.  Returns the index in every lane.
template <typename TE>
__device__ int block_search(const RowDesc &dp, const RowDesc &dq, int residual, float c,
                            const TE *gp, const TE *gq, int bs, int be, float t, float &margin) {
  const int lane = threadIdx.x & 31;
  float base_sum = 0.f;
  int result = -1, lastpos = -1;
  margin = 0.f;
  for (int rb = bs; rb < be && result < 0; rb += 256) {
    const int base = rb + lane * 8;
    float w[8];
    float s = 0.f;
    int lp = -1;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int v = base + e;
      float x = 0.f;
      if (v < be) {
        const float zp = dp.onehot ? 0.f : to_f32(gp[v]);
        const float zq = (residual && !dq.onehot) ? to_f32(gq[v]) : 0.f;
        x = weight(dp, dq, residual, c, zp, zq, v);
      }
      w[e] = x;
      s += x;
      if (x > 0.f) lp = v;
    }
    float incl = s;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const float u = __shfl_up_sync(0xFFFFFFFFu, incl, off);
      if (lane >= off) incl += u;
    }
    float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
    if (lane == 0) excl = 0.f;
    lastpos = max(lastpos, warp_max_i(lp));
    const unsigned hit = __ballot_sync(0xFFFFFFFFu, base_sum + incl > t);
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
          if (found < 0 && w[e] > 0.f && run > t) {
            found = base + e;
            mg = fminf(t - prev, run - t);
          }
        }
        if (found < 0) found = lp;
      }
      result = __shfl_sync(0xFFFFFFFFu, found, first);
      margin = __shfl_sync(0xFFFFFFFFu, mg, first);
    }
    base_sum += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  if (result < 0 || t == INFINITY) margin = 0.f;
  return result >= 0 ? result : lastpos;
}

// Draw the unit's token from the block totals of its held distribution
// (warp 0; returns the token in every lane of warp 0).
template <typename TE>
__device__ int draw_from_blocks(const Params &P, const UnitInfo &u, const DrawState &ds,
                                float Z, float &margin) {
  const int lane = threadIdx.x & 31;
  const int C = P.cluster, sb = P.slice_blocks;
  const int nb = C * sb;
  const float *blk = P.wblk + static_cast<long long>(u.seq * P.ups + u.node) * nb;
  const float t = unit_uniform(P, u.seq, u.node, 1) * Z;
  // every lane owns a contiguous run of blocks
  const int per = (nb + 31) / 32;
  const int b0 = lane * per, b1 = min(nb, b0 + per);
  float seg = 0.f;
  int lastpos_blk = -1;
  for (int b = b0; b < b1; ++b) {
    const float x = __ldcg(blk + b);
    seg += x;
    if (x > 0.f) lastpos_blk = b;
  }
  float incl = seg;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float v = __shfl_up_sync(0xFFFFFFFFu, incl, off);
    if (lane >= off) incl += v;
  }
  float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
  if (lane == 0) excl = 0.f;
  const unsigned hit = __ballot_sync(0xFFFFFFFFu, incl > t);
  int ob = -1;
  float trel = INFINITY;
  if (hit) {
    const int first = __ffs(hit) - 1;
    int found = -1;
    float tr = INFINITY;
    if (lane == first) {
      float run = excl;
      for (int b = b0; b < b1; ++b) {
        const float x = __ldcg(blk + b);
        if (run + x > t) {
          found = b;
          tr = t - run;
          break;
        }
        run += x;
      }
      if (found < 0) {
        found = lastpos_blk;
        tr = INFINITY;
      }
    }
    ob = __shfl_sync(0xFFFFFFFFu, found, first);
    trel = __shfl_sync(0xFFFFFFFFu, tr, first);
  }
  if (ob < 0) {
    ob = warp_max_i(lastpos_blk);
    trel = INFINITY;
  }
  int bs, be;
  block_range(P, ob / sb, ob % sb, sizeof(TE), bs, be);
  const TE *gp = static_cast<const TE *>(row_ptr(P.target, u.prow, P.ld_t, sizeof(TE)));
  const TE *gq = static_cast<const TE *>(row_ptr(P.draft, u.qrow, P.ld_d, sizeof(TE)));
  const int residual = ds.c_cur > 0.f;
  return block_search<TE>(ds.dp, ds.dq, residual, residual ? ds.c_cur : 0.f, gp, gq, bs, be,
                          trel, margin);
}

// ---------------------------------------------------------------------------
// finishing steps (compute threads of the CTA that completed a counter)
// ---------------------------------------------------------------------------

// All stats slices of `unit` are in: merge, decide or queue the first round.
template <typename TE>
__device__ void decide_unit(const Params &P, int unit, Ctl3 &ctl) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int C = P.cluster, V = P.V;
  const UnitInfo u = decode_unit(P, unit);
  if (warp == 0) {
    for (int row = 0; row < 2; ++row) {
      if (row == 1 && !u.load_q) break;
      const int arg = row == 0 ? u.p_arg : u.q_arg;
      const float kk = row == 0 ? u.kp : u.kq;
      Partial o;
      o.m = -INFINITY;
      o.S = 0.f;
      o.av = -INFINITY;
      o.ai = INT_MAX;
      o.flags = 0;
      for (int r = lane; r < C; r += 32) {
        const SlicePartial *sp = P.partials + (static_cast<long long>(unit) * C + r) * 2 + row;
        const float m2 = __ldcg(&sp->m), S2 = __ldcg(&sp->S), v2 = __ldcg(&sp->av);
        const int i2 = __ldcg(&sp->ai), f2 = __ldcg(&sp->flags);
        o.flags |= f2;
        if (arg) argmax_merge(o.av, o.ai, v2, i2);
        else online_merge(o.m, o.S, m2, S2, kk);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float m2 = __shfl_xor_sync(0xFFFFFFFFu, o.m, off);
        const float S2 = __shfl_xor_sync(0xFFFFFFFFu, o.S, off);
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, o.av, off);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, o.ai, off);
        o.flags |= __shfl_xor_sync(0xFFFFFFFFu, o.flags, off);
        if (arg) argmax_merge(o.av, o.ai, v2, i2);
        else online_merge(o.m, o.S, m2, S2, kk);
      }
      if (lane == 0) ctl.merged[row] = o;
    }
  }
  csync();
  DrawState ds;
  ds.flags = 0u;
  int need_fallback[2] = {0, 0};
  for (int row = 0; row < 2; ++row) {
    RowDesc d;
    d.m = 0.f;
    d.flags = 0u;
    d.thr = -INFINITY;
    if (row == 1 && !u.load_q) {
      d.onehot = 1;
      d.a = 0;
      d.k = d.nmk = d.invS = 0.f;
      ds.dq = d;
      break;
    }
    const int arg = row == 0 ? u.p_arg : u.q_arg;
    const int tbad = row == 0 ? u.tp_bad : u.tq_bad;
    const float kk = row == 0 ? u.kp : u.kq;
    const Partial o = ctl.merged[row];
    if (o.flags & 4) ds.flags |= SPEC_FLAG_TIMEOUT;
    if (arg) {
      d.onehot = 1;
      d.a = o.ai == INT_MAX ? 0 : o.ai;
      d.k = d.nmk = d.invS = 0.f;
      if (tbad || (o.flags & 3) || o.ai == INT_MAX) d.flags = SPEC_FLAG_NONFINITE;
    } else {
      const float M = o.m, S = o.S;
      const bool bad = (o.flags & 3) || !(M > -INFINITY) || M == INFINITY || !(S > 0.f) ||
                       S == INFINITY || S != S;
      d.onehot = 0;
      d.a = 0;
      d.k = kk;
      d.m = M;
      d.nmk = -M * kk;
      d.invS = 1.f / S;
      if (bad) {
        need_fallback[row] = 1;
        d.onehot = 1;
        d.flags = SPEC_FLAG_NONFINITE;
      }
    }
    if (row == 0) ds.dp = d; else ds.dq = d;
  }
  csync();
  // finite-argmax fallback for non-finite sampling rows (rare): re-read the row
  for (int row = 0; row < 2; ++row) {
    if (!need_fallback[row]) continue;
    RowAcc a;
    acc_init(a);
    const TE *gr = static_cast<const TE *>(row_ptr(row == 0 ? P.target : P.draft,
                                                   row == 0 ? u.prow : u.qrow,
                                                   row == 0 ? P.ld_t : P.ld_d, sizeof(TE)));
    for (int v = tid; v < V; v += kThreads) acc_scalar_argmax(a, to_f32(gr[v]), v);
    block_argmax(a.bv, a.bi, a.fl, ctl.rs);
    if (row == 0) ds.dp.a = a.bi == INT_MAX ? 0 : a.bi;
    else ds.dq.a = a.bi == INT_MAX ? 0 : a.bi;
  }
  if (tid == 0) {
    ds.flags |= ds.dp.flags;
    ds.c = 0.f;
    ds.c_cur = 0.f;
    ds.W_cur = 0.f;
    ds.round = 0;
    ds.blocks_c_valid = 0;
    ds.n_res = 0;
    int child = u.has_children
                    ? (P.mode == kModeChain ? u.node + 1 : __ldg(P.first_child + unit))
                    : -1;
    ds.child = child;
    if (ds.dp.onehot) {
      // greedy rule: accept the first child equal to the argmax; q is not used
      int next = -1;
      for (; child >= 0; child = next_child_1(P, u.seq, u.node, child)) {
        const int x = child_token(P, u.seq, u.node, child);
        if (x < 0 || x >= V) ds.flags |= SPEC_FLAG_BAD_TOKEN;
        if (x == ds.dp.a) {
          next = child;
          break;
        }
      }
      publish_unit(P, unit, u.node, next, next < 0 ? ds.dp.a : -1, ds.flags, ds.dp, ds.dq, 0.f,
                   0.f, (next < 0 && u.has_children) ? 1 : 0);
    } else {
      if (u.has_children) ds.flags |= ds.dq.flags;
      bool rejected = false;
      const int acc = child >= 0 ? test_children<TE>(P, u, ds, child, true, rejected) : -1;
      if (acc >= 0) {
        publish_unit(P, unit, u.node, acc, -1, ds.flags, ds.dp, ds.dq, 0.f, 0.f, 0);
      } else {
        ds.c = rejected ? 1.f : 0.f;  // residual after the rejection, or the bonus draw from p
        enqueue_round(P, unit, ds);
      }
    }
  }
  csync();
}

// All weight slices of a round of `unit` are in: finish the round.
template <typename TE>
__device__ void finish_round(const Params &P, int unit, Ctl3 &ctl) {
  const int tid = threadIdx.x;
  const int C = P.cluster;
  const UnitInfo u = decode_unit(P, unit);
  DrawState ds;
  bool draw = false;
  float Z = 0.f;
  if (tid == 0) {
    ds = load_dstate(P.dstate + unit);
    P.w_done[unit] = 0u;
    float W = 0.f;
    for (int r = 0; r < C; ++r) W += __ldcg(P.wpart + static_cast<long long>(unit) * C + r);
    bool more = false;
    if (ds.c > 0.f) {  // a residual candidate [p - c q]_+
      if (W > 0.f) {
        ds.c_cur = ds.c;
        ds.W_cur = W;
        ds.blocks_c_valid = 1;
        ds.n_res += 1;
      } else {
        ds.flags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
        ds.blocks_c_valid = 0;
      }
      // the next sibling, tested with the distribution now held
      int child = next_child_1(P, u.seq, u.node, ds.child);
      if (child >= 0) {
        bool rejected = false;
        const int acc = test_children<TE>(P, u, ds, child, true, rejected);
        if (acc >= 0) {
          publish_unit(P, unit, u.node, acc, -1, ds.flags, ds.dp, ds.dq, 0.f, 0.f, 0);
          ctl.decision = 0;
          more = true;  // nothing left to do
        } else {
          ds.c = ds.c_cur > 0.f ? ds.c_cur + ds.W_cur : 1.f;
          enqueue_round(P, unit, ds);
          more = true;
        }
      }
      if (!more) {
        if (ds.blocks_c_valid) {
          Z = ds.W_cur;
          draw = true;
        } else {  // block totals of the held distribution are needed again
          ds.c = ds.c_cur;
          enqueue_round(P, unit, ds);
        }
      }
    } else {  // the weights were p itself: the bonus draw or the draw after a degenerate residual
      Z = W;
      draw = true;
    }
    ctl.decision = draw ? 1 : 0;
    ctl.trel = Z;
    ctl.ds_share = ds;  // hand the state to warp 0
  }
  csync();
  if (ctl.decision && tid < 32) {
    const DrawState dsw = ctl.ds_share;
    float margin;
    const int tok = draw_from_blocks<TE>(P, u, dsw, ctl.trel, margin);
    if (tid == 0) {
      const int residual = dsw.c_cur > 0.f;
      const float c = residual ? dsw.c_cur : 0.f;
      publish_unit(P, unit, u.node, -1, tok, dsw.flags, dsw.dp, dsw.dq, c, ctl.trel,
                   u.has_children ? 2 : 0, margin < kRefineGuard * (1.f + c) ? 1 : 0,
                   residual ? dsw.n_res : 0);
    }
  }
  csync();
}

// ---------------------------------------------------------------------------
// the streaming kernel
// ---------------------------------------------------------------------------

template <typename TE>
__global__ void __launch_bounds__(kBlockThreads, 3) stream_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Ctl3 &ctl = *reinterpret_cast<Ctl3 *>(smem_raw);
  unsigned char *ring = smem_raw + P.data_off;
  constexpr int PE = 16 / sizeof(TE);
  const int C = P.cluster;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int NS = P.ring;
  const int cvec = P.slot_bytes / 16;
  const int chunks = P.chunks;
  const long long n_tasks = static_cast<long long>(P.n_units) * C;

  if (tid == 0) {
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl.full[s], 1);
      mbar_init(&ctl.empty[s], 1);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  }
  __syncthreads();

  if (warp == kProducerWarp) {
    // ---- the scheduler: claim tasks and stream their chunks
    if (lane == 0) {
      long long item = 0;
      int k = 0;
      long long stats_next = blockIdx.x;
      long long idle_since = -1;
      // one queue ticket at a time: the scheduler that drew ticket i runs the
      // i-th weight task queued, as soon as it is there; until then it keeps
      // streaming its own stats tasks (no spinning on the shared counters)
      long long ticket = atomicAdd(P.wq_ctr + 0, 1u);
      for (;;) {
        TaskInfo ti;
        ti.round = 0;
        ti.bits = 0;
        ti.kp = ti.kq = ti.c = 0.f;
        int rows = 0;
        long long prow = 0, qrow = 0;
        bool have = false;
        if (ticket >= 0 && ticket < P.wq_cap) {
          const volatile int *e = reinterpret_cast<const volatile int *>(P.wq + ticket);
          if (e[3] == static_cast<int>(P.epoch)) {
            __threadfence();
            const int unit = e[0], slice = e[1], round = e[2];
            const DrawState ds = load_dstate(P.dstate + unit);
            const UnitInfo u = decode_unit(P, unit);
            ti.type = kTaskWeights;
            ti.unit = unit;
            ti.slice = slice;
            ti.round = round;
            ti.c = ds.c;
            ti.dp = ds.dp;
            ti.dq = ds.dq;
            rows = ds.c > 0.f ? 2 : 1;
            prow = u.prow;
            qrow = u.qrow;
            have = true;
            ticket = atomicAdd(P.wq_ctr + 0, 1u);
          }
        }
        if (!have && stats_next < n_tasks) {
          const int unit = static_cast<int>(stats_next / C);
          const UnitInfo u = decode_unit(P, unit);
          ti.type = kTaskStats;
          ti.unit = unit;
          ti.slice = static_cast<int>(stats_next % C);
          ti.bits = (u.p_arg ? 1 : 0) | (u.q_arg ? 2 : 0) | (u.tp_bad ? 4 : 0) |
                    (u.tq_bad ? 8 : 0) | (u.load_q ? 16 : 0) | (u.has_children ? 32 : 0);
          ti.kp = u.kp;
          ti.kq = u.kq;
          rows = u.load_q ? 2 : 1;
          prow = u.prow;
          qrow = u.qrow;
          stats_next += gridDim.x;
          have = true;
        }
        if (!have) {
          // nothing to stream: finish once every unit is complete
          if (ld_volatile(P.wq_ctr + 2) >= static_cast<uint32_t>(P.n_units)) break;
          if (idle_since < 0) idle_since = global_ns();
          if (global_ns() - idle_since > kPollLimitNs) break;
          __nanosleep(128);
          continue;
        }
        idle_since = -1;
        const SliceGeo g = slice_geo(P, ti.slice, sizeof(TE));
        for (int row = 0; row < rows; ++row) {
          const TE *src = static_cast<const TE *>(
              row_ptr(row == 0 ? P.target : P.draft, row == 0 ? prow : qrow,
                      row == 0 ? P.ld_t : P.ld_d, sizeof(TE))) + g.v0;
          for (int cc = 0; cc < chunks; ++cc, ++item) {
            const int slot = static_cast<int>(item % NS);
            const long long use = item / NS;
            if (use > 0) mbar_wait_bounded(&ctl.empty[slot], static_cast<uint32_t>((use - 1) & 1));
            if (row == 0 && cc == 0) ctl.tinfo[k % kMaxRing] = ti;  // published by the arrive
            const int vb = min(g.nvec, cc * cvec), ve = min(g.nvec, (cc + 1) * cvec);
            const uint32_t bytes = static_cast<uint32_t>(ve - vb) * 16u;
            mbar_arrive_expect_tx(&ctl.full[slot], bytes);
            if (bytes)
              bulk_g2s_plain(ring + static_cast<size_t>(slot) * P.slot_bytes, src + vb * PE, bytes,
                             &ctl.full[slot]);
          }
        }
        ++k;
      }
      // tell the compute threads to stop: an empty item carrying the end marker
      const int slot = static_cast<int>(item % NS);
      const long long use = item / NS;
      if (use > 0) mbar_wait_bounded(&ctl.empty[slot], static_cast<uint32_t>((use - 1) & 1));
      TaskInfo end;
      end.type = kTaskEnd;
      end.unit = end.slice = end.round = end.bits = 0;
      ctl.tinfo[k % kMaxRing] = end;
      mbar_arrive_expect_tx(&ctl.full[slot], 0u);
    }
    __syncwarp();
  } else {
    // ---- compute threads: process tasks in the order they were streamed
    long long item = 0;
    for (int k = 0;; ++k) {
      const int slot0 = static_cast<int>(item % NS);
      int timeout = 0;
      if (!mbar_wait_bounded(&ctl.full[slot0], static_cast<uint32_t>((item / NS) & 1))) {
        timeout = 4;
        mbar_wait_bounded(&ctl.full[slot0], static_cast<uint32_t>((item / NS) & 1));
      }
      const TaskInfo ti = ctl.tinfo[k % kMaxRing];
      if (ti.type == kTaskEnd) break;
      const int unit = ti.unit, r = ti.slice;
      const SliceGeo g = slice_geo(P, r, sizeof(TE));
      const int seq = unit / P.ups, node = unit % P.ups;
      long long prow, qrow;
      if (P.mode == kModeChain) {
        prow = static_cast<long long>(seq) * (P.gamma + 1) + node;
        qrow = static_cast<long long>(seq) * P.gamma + node;
      } else {
        prow = static_cast<long long>(seq) * P.ups + node;
        qrow = prow;
      }
      const TE *gp = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE))) + g.v0;
      const TE *gq = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE))) + g.v0;

      if (ti.type == kTaskStats) {
        const int p_arg = ti.bits & 1, q_arg = ti.bits & 2;
        const int rows = (ti.bits & 16) ? 2 : 1;
        RowAcc acc[2];
        acc_init(acc[0]);
        acc_init(acc[1]);
        for (int row = 0; row < rows; ++row) {
          const int arg = row == 0 ? p_arg : q_arg;
          const float kk = row == 0 ? ti.kp : ti.kq;
          RowAcc &a = acc[row];
          for (int cc = 0; cc < chunks; ++cc, ++item) {
            const int slot = static_cast<int>(item % NS);
            const uint32_t phase = static_cast<uint32_t>((item / NS) & 1);
            if (!(row == 0 && cc == 0) && !mbar_wait_bounded(&ctl.full[slot], phase)) {
              timeout = 4;
              mbar_wait_bounded(&ctl.full[slot], phase);
            }
            const TE *s = reinterpret_cast<const TE *>(ring + static_cast<size_t>(slot) * P.slot_bytes);
            const int nv = max(0, min(cvec, g.nvec - cc * cvec));
            if (arg) {
              RowAcc tt;
              acc_init(tt);
              stage_argmax<TE>(s, 0, nv * PE, g.v0 + cc * cvec * PE, tt);
              a.fl |= tt.fl;
              argmax_merge(a.bv, a.bi, tt.bv, tt.bi);
            } else {
              stage_softmax(s, 0, nv, kk, a);
            }
            csync();  // every compute thread is done with the slot
            if (tid == 0) mbar_arrive(&ctl.empty[slot]);
          }
          if (tid == 0) {  // the ragged tail the bulk copies skip
            const TE *gr = row == 0 ? gp : gq;
            for (int e = g.nvec * PE; e < g.len; ++e) {
              if (arg) acc_scalar_argmax(a, to_f32(gr[e]), g.v0 + e);
              else acc_scalar_softmax(a, to_f32(gr[e]), kk);
            }
          }
          a.fl |= timeout;
        }
        for (int row = 0; row < rows; ++row) {
          RowAcc &a = acc[row];
          const int arg = row == 0 ? p_arg : q_arg;
          if (arg) block_argmax(a.bv, a.bi, a.fl, ctl.rs);
          else block_online(a.m, a.S, a.fl, row == 0 ? ti.kp : ti.kq, ctl.rs);
          if (tid == 0) {
            SlicePartial sp;
            sp.m = a.m;
            sp.S = a.S;
            sp.av = a.bv;
            sp.ai = a.bi;
            sp.flags = a.fl;
            sp.pad[0] = sp.pad[1] = sp.pad[2] = 0;
            P.partials[(static_cast<long long>(unit) * C + r) * 2 + row] = sp;
          }
        }
        if (tid == 0) {
          __threadfence();
          const unsigned prev = atomicAdd(P.unit_done + unit, 1u);
          ctl.is_last = prev == static_cast<unsigned>(C - 1);
          if (ctl.is_last) __threadfence();
        }
        csync();
        if (ctl.is_last) decide_unit<TE>(P, unit, ctl);
      } else {
        // weight task: per-block totals of [p - c q]_+ (or p) over the slice
        const int residual = ti.c > 0.f;
        const RowDesc dp = ti.dp, dq = ti.dq;
        const float c = ti.c;
        const int bl = ((cvec * PE + kBlocksPerChunk - 1) / kBlocksPerChunk + 7) / 8 * 8;
        const bool fast = sizeof(TE) == 2 && !dp.onehot && dp.thr == -INFINITY &&
                          (!residual || (!dq.onehot && dq.thr == -INFINITY));
        float *blk_out = P.wblk + static_cast<long long>(unit) * C * P.slice_blocks +
                         static_cast<long long>(r) * P.slice_blocks;
        for (int cc = 0; cc < chunks; ++cc) {
          // the p chunk and, for residual weights, the q chunk of the same range
          const long long ip = item + cc;
          const long long iq = item + chunks + cc;
          const int sp_slot = static_cast<int>(ip % NS);
          const int sq_slot = static_cast<int>(iq % NS);
          if (!(cc == 0) && !mbar_wait_bounded(&ctl.full[sp_slot], static_cast<uint32_t>((ip / NS) & 1)))
            timeout = 4;
          if (residual && !mbar_wait_bounded(&ctl.full[sq_slot], static_cast<uint32_t>((iq / NS) & 1)))
            timeout = 4;
          const TE *sp = reinterpret_cast<const TE *>(ring + static_cast<size_t>(sp_slot) * P.slot_bytes);
          const TE *sq = reinterpret_cast<const TE *>(ring + static_cast<size_t>(sq_slot) * P.slot_bytes);
          const int cn = max(0, min(cvec, g.nvec - cc * cvec)) * PE;
          const int vbase = g.v0 + cc * cvec * PE;
          for (int half = 0; half < 2; ++half) {
            const int bi = warp + half * kWarps;
            const int bs = min(cn, bi * bl), be = min(cn, bs + bl);
            float a = 0.f;
            if (fast) {
              const uint64_t kp2 = pack2(dp.k, dp.k), np2 = pack2(dp.nmk, dp.nmk);
              const uint64_t ia2 = pack2(dp.invS, dp.invS);
              const uint64_t kq2 = pack2(dq.k, dq.k), nq2 = pack2(dq.nmk, dq.nmk);
              const uint64_t ib2 = pack2(dq.invS, dq.invS), nc2 = pack2(-c, -c);
              for (int o = bs + lane * 8; o < be; o += 256) {
                const uint4 wp = *reinterpret_cast<const uint4 *>(sp + o);
                const uint32_t pw[4] = {wp.x, wp.y, wp.z, wp.w};
                if (!residual) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    float a0, a1;
                    unpack2(fmul2(ex2_pair(ffma2(bf16x2_to_pair(pw[j]), kp2, np2)), ia2), a0, a1);
                    a += a0 + a1;
                  }
                } else {
                  const uint4 wq = *reinterpret_cast<const uint4 *>(sq + o);
                  const uint32_t qw[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    const uint64_t pv = fmul2(ex2_pair(ffma2(bf16x2_to_pair(pw[j]), kp2, np2)), ia2);
                    const uint64_t qv = fmul2(ex2_pair(ffma2(bf16x2_to_pair(qw[j]), kq2, nq2)), ib2);
                    float d0, d1;
                    unpack2(ffma2(qv, nc2, pv), d0, d1);
                    a += fmaxf(d0, 0.f) + fmaxf(d1, 0.f);
                  }
                }
              }
            } else {
              for (int o = bs + lane; o < be; o += 32) {
                const float zp = dp.onehot ? 0.f : to_f32(sp[o]);
                const float zq = (residual && !dq.onehot) ? to_f32(sq[o]) : 0.f;
                a += weight(dp, dq, residual, c, zp, zq, vbase + o);
              }
            }
            a = warp_sum(a);
            if (lane == 0) ctl.btot[cc * kBlocksPerChunk + bi] = a;
          }
        }
        item += static_cast<long long>(chunks) * (residual ? 2 : 1);
        csync();  // every compute thread is done with the task's slots
        if (tid == 0) {
          for (long long i = item - static_cast<long long>(chunks) * (residual ? 2 : 1); i < item; ++i)
            mbar_arrive(&ctl.empty[static_cast<int>(i % NS)]);
          // the ragged tail, then the slice total in index order
          float tail = 0.f;
          for (int e = g.nvec * PE; e < g.len; ++e)
            tail += weight(dp, dq, residual, c, to_f32(gp[e]), residual ? to_f32(gq[e]) : 0.f,
                           g.v0 + e);
          const int nblk = chunks * kBlocksPerChunk;
          float tot = 0.f;
          for (int b = 0; b < nblk; ++b) {
            blk_out[b] = ctl.btot[b];
            tot += ctl.btot[b];
          }
          blk_out[nblk] = tail;
          tot += tail;
          P.wpart[static_cast<long long>(unit) * C + r] = tot;
          __threadfence();
          const unsigned prev = atomicAdd(P.w_done + unit, 1u);
          ctl.is_last = prev == static_cast<unsigned>(C - 1);
          if (ctl.is_last) __threadfence();
        }
        csync();
        if (ctl.is_last) finish_round<TE>(P, unit, ctl);
      }
    }
  }
  __syncthreads();
}

// ---------------------------------------------------------------------------
// stitching the paths
// ---------------------------------------------------------------------------

// One warp per chain: the first rejected position j by a ballot.  Block 0
// also clears the queue counters for the next call.
__global__ void __launch_bounds__(kThreads) chain_combine_kernel(const Params P) {
  if (blockIdx.x == 0 && threadIdx.x < 3 && P.wq_ctr) P.wq_ctr[threadIdx.x] = 0u;
  const int seq = blockIdx.x * kWarps + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (seq >= P.nseq) return;
  const long long ubase = static_cast<long long>(seq) * P.ups;
  int j = -1;
  for (int base = 0; base <= P.gamma && j < 0; base += 32) {
    const int i = base + lane;
    const bool stop = i <= P.gamma && P.outs[ubase + i].next < 0;
    const unsigned b = __ballot_sync(0xFFFFFFFFu, stop);
    if (b) j = base + __ffs(b) - 1;
  }
  uint32_t f = 0u;
  for (int i = lane; i <= j; i += 32) f |= P.outs[ubase + i].flags;
  f = warp_or(f);
  const int jtok = P.outs[ubase + j].token;
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
    queue_refine(P, seq, ubase + j, j, P.outs[ubase + j].near);
  }
}

// One CTA per tree: validate the links, depths by pointer jumping, then walk
// the accepted children from the root.  Block 0 also clears the queue
// counters for the next call.
__global__ void __launch_bounds__(kThreads) tree_combine_kernel(const Params P) {
  extern __shared__ int tsm[];
  __shared__ uint32_t red[kWarps];
  if (blockIdx.x == 0 && threadIdx.x < 3 && P.wq_ctr) P.wq_ctr[threadIdx.x] = 0u;
  const int seq = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int N = P.ups;
  const long long ubase = static_cast<long long>(seq) * N;
  const int32_t *par = P.parent + ubase;
  int *anc = tsm;
  int *dep = tsm + N;
  uint32_t bad = 0u;
  for (int n = tid; n < N; n += kThreads) {
    const int a = __ldg(par + n);
    if (n == 0 ? a != -1 : !(a >= 0 && a < n)) bad = 1u;
    anc[n] = n == 0 ? 0 : a;
    dep[n] = n == 0 ? 0 : 1;
  }
  bad = warp_or(bad);
  if (lane == 0) red[warp] = bad;
  __syncthreads();
  bad = 0u;
  for (int w = 0; w < kWarps; ++w) bad |= red[w];
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
    if (lane == 0) red[warp] = deep;
    __syncthreads();
    deep = 0u;
    for (int w = 0; w < kWarps; ++w) deep |= red[w];
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
    return;
  }
  if (tid == 0) {
    int cur = 0, k = 0;
    uint32_t f = P.outs[ubase].flags;
    P.out_path[obase] = 0;
    int nx = P.outs[ubase].next;
    while (nx > cur && nx < N && k < P.max_depth) {
      ++k;
      cur = nx;
      P.out_path[obase + k] = cur;
      P.out_tokens[obase + k - 1] = __ldg(P.tokens + ubase + cur);
      f |= P.outs[ubase + cur].flags;
      nx = P.outs[ubase + cur].next;
    }
    P.out_tokens[obase + k] = P.outs[ubase + cur].token;
    for (int i = k + 1; i < width; ++i) {
      P.out_path[obase + i] = -1;
      P.out_tokens[obase + i] = -1;
    }
    P.out_num[seq] = k;
    if (P.out_flags) P.out_flags[seq] = f;
    P.final_unit[seq] = static_cast<int>(ubase + cur);
    queue_refine(P, seq, ubase + cur, k, P.outs[ubase + cur].near);
  }
}

// First child of every tree node (-1 for leaves); children are the nodes c
// with 0 <= parent[c] < c.
__global__ void __launch_bounds__(kThreads) tree_first_child_kernel(const int32_t *parent, int N,
                                                                    int32_t *first_child) {
  extern __shared__ int fc[];
  // a kernel launched behind this one with programmatic serialisation may
  // start now; it waits for these results before it reads them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const long long base = static_cast<long long>(blockIdx.x) * N;
  for (int n = threadIdx.x; n < N; n += kThreads) fc[n] = INT_MAX;
  __syncthreads();
  for (int c = threadIdx.x; c < N; c += kThreads) {
    const int p = __ldg(parent + base + c);
    if (c > 0 && p >= 0 && p < c) atomicMin(&fc[p], c);
  }
  __syncthreads();
  for (int n = threadIdx.x; n < N; n += kThreads)
    first_child[base + n] = fc[n] == INT_MAX ? -1 : fc[n];
}

// ---------------------------------------------------------------------------
// launchers
// ---------------------------------------------------------------------------

template <typename TE>
cudaError_t launch_stream_t(const Params &P, size_t smem, cudaStream_t stream) {
  auto kern = stream_kernel<TE>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  // resident CTAs per SM for this footprint (cached per shared-memory size)
  static std::mutex mu;  // guards the cache below across host threads
  static int cache_key[16][2];
  static int cache_val[16];
  static int cache_n = 0;
  int per_sm = 0;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < cache_n; ++i)
    if (cache_key[i][0] == static_cast<int>(smem) && cache_key[i][1] == static_cast<int>(sizeof(TE)))
      per_sm = cache_val[i];
  if (per_sm == 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kBlockThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    if (cache_n < 16) {
      cache_key[cache_n][0] = static_cast<int>(smem);
      cache_key[cache_n][1] = static_cast<int>(sizeof(TE));
      cache_val[cache_n] = per_sm;
      ++cache_n;
    }
  }
  int dev = 0, sms = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long n_tasks = static_cast<long long>(P.n_units) * P.cluster;
  long long grid = static_cast<long long>(per_sm) * sms;
  if (grid > n_tasks) grid = n_tasks;
  Params Pc = P;
  void *args[] = {&Pc};
  // cooperative: every CTA resident, so the schedulers' final polling always ends
  return cudaLaunchCooperativeKernel(reinterpret_cast<void *>(kern),
                                     dim3(static_cast<unsigned>(grid)), dim3(kBlockThreads), args,
                                     smem, stream);
}

cudaError_t launch_stream(const Params &P, int esize, size_t smem, cudaStream_t stream) {
  cudaError_t e = esize == 2 ? launch_stream_t<uint16_t>(P, smem, stream)
                             : launch_stream_t<float>(P, smem, stream);
  if (e != cudaSuccess) return e;
  if (P.mode == kModeChain) {
    chain_combine_kernel<<<(P.nseq + kWarps - 1) / kWarps, kThreads, 0, stream>>>(P);
  } else {
    const size_t tsm = 2 * sizeof(int) * static_cast<size_t>(P.ups);
    if (tsm > 48 * 1024) {
      e = cudaFuncSetAttribute(tree_combine_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(tsm));
      if (e != cudaSuccess) return e;
    }
    tree_combine_kernel<<<P.nseq, kThreads, tsm, stream>>>(P);
  }
  return cudaGetLastError();
}

cudaError_t launch_first_child(const int32_t *parent, int T, int N, int32_t *first_child,
                               cudaStream_t stream) {
  tree_first_child_kernel<<<T, kThreads, sizeof(int) * static_cast<size_t>(N), stream>>>(
      parent, N, first_child);
  return cudaGetLastError();
}

}  // namespace sv
