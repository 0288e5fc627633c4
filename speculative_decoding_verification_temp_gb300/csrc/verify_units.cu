// Resident verification kernel (every CTA keeps its slice of the unit's row
// pair in shared memory for the whole unit) and the residual-output kernel.
// Used for launches with top-k filtering or rows that are not 16-byte aligned;
// see verify_units.cuh for the design and verify_stream.cu for the streaming
// kernel that serves the other launches.
#include "ops.cuh"

namespace sv {

// Cluster sum of the current draw weights; fills ctl.parts (per-CTA totals in
// rank order) and returns the total.  Cluster-collective.
template <typename TE>
__device__ float cluster_total(const RowDesc &dp, const RowDesc &dq, int residual, float c,
                               const TE *sp, const TE *sq, int v0, int len, Ctl &ctl,
                               cg::cluster_group &cluster, int C, int &xround) {
  float acc = slice_total<TE>(dp, dq, residual, c, sp, sq, v0, len);
  acc = block_sum(acc, ctl.rs);
  const int buf = xround & 1;
  ++xround;
  if (threadIdx.x == 0) ctl.wx[buf][0] = acc;
  cluster_sync_all();
  if (threadIdx.x < C) ctl.parts[threadIdx.x] = cluster.map_shared_rank(&ctl.wx[buf][0], threadIdx.x)[0];
  __syncthreads();
  float total = 0.f;
  for (int r = 0; r < C; ++r) total += ctl.parts[r];
  return total;
}

// ---------------------------------------------------------------------------
// the unit kernel
// ---------------------------------------------------------------------------

template <typename TE, bool kVec>
__global__ void __launch_bounds__(kThreads) unit_kernel(const Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  Ctl &ctl = *reinterpret_cast<Ctl *>(smem_raw);
  TE *sp = reinterpret_cast<TE *>(smem_raw + P.data_off);
  TE *sq = sp + P.slice;
  cg::cluster_group cluster = cg::this_cluster();
  constexpr int PV = Elem<TE>::kPerVec;
  const int C = P.cluster;
  const int rank = static_cast<int>(cluster.block_rank());
  const int unit = blockIdx.x / C;
  const int seq = unit / P.ups, node = unit % P.ups;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
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

  int child = next_child(P, seq, node, -1, ctl.rs);
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
  const TE *gp_row = static_cast<const TE *>(row_ptr(P.target, prow, P.ld_t, sizeof(TE)));
  const TE *gq_row = static_cast<const TE *>(row_ptr(P.draft, qrow, P.ld_d, sizeof(TE)));
  const TE *gp = gp_row + v0;
  const TE *gq = gq_row + v0;

  // ---- 1. issue the slice loads
  const int nvec = kVec ? (len * static_cast<int>(sizeof(TE))) / 16 : 0;
  const int nvs = (nvec + kStages - 1) / kStages;
  if (kVec) {
    if (tid == 0) {
      for (int s = 0; s < kStages; ++s) mbar_init(&ctl.bar[s], 1);
      asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      uint64_t policy;
      asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(policy));
      for (int s = 0; s < kStages; ++s) {
        const int vb = min(nvec, s * nvs), ve = min(nvec, (s + 1) * nvs);
        const uint32_t bytes = static_cast<uint32_t>(ve - vb) * 16u;
        mbar_arrive_expect_tx(&ctl.bar[s], load_q ? 2u * bytes : bytes);
        if (bytes) {
          bulk_g2s(sp + vb * PV, gp + vb * PV, bytes, &ctl.bar[s], policy);
          if (load_q) bulk_g2s(sq + vb * PV, gq + vb * PV, bytes, &ctl.bar[s], policy);
        }
      }
      for (int e = nvec * PV; e < len; ++e) {
        sp[e] = gp[e];
        if (load_q) sq[e] = gq[e];
      }
    }
  } else {
    for (int e = tid; e < len; e += kThreads) {
      sp[e] = gp[e];
      if (load_q) sq[e] = gq[e];
    }
  }
  // gather the first child's logits (thread 0) while the slices stream in
  float pre_zp = 0.f, pre_zq = 0.f;
  if (tid == 0 && has_children) {
    const int x = child_token(P, seq, node, child);
    if (x >= 0 && x < V) {
      pre_zp = to_f32(gp_row[x]);
      if (load_q) pre_zq = to_f32(gq_row[x]);
    }
  }
  __syncthreads();

  // ---- 2. row statistics
  const bool topk_p = !p_arg && kp_raw > 0 && kp_raw < V;
  const bool topk_q = load_q && !q_arg && kq_raw > 0 && kq_raw < V;
  float thr_p = -INFINITY, thr_q = -INFINITY;
  const float kpv = p_arg ? 0.f : kLog2e / Tp;
  const float kqv = q_arg ? 0.f : kLog2e / Tq;
  RowAcc ap, aq;
  acc_init(ap);
  acc_init(aq);
  int tflag = 0;
  if (!(topk_p || topk_q)) {
    for (int s = 0; s < kStages; ++s) {
      const int vb = min(nvec, s * nvs), ve = min(nvec, (s + 1) * nvs);
      if (kVec && !mbar_wait_bounded(&ctl.bar[s], 0)) tflag = 4;
      if (!kVec && s > 0) break;
      const int eb = kVec ? vb * PV : 0, ee = kVec ? ve * PV : len;
      if (p_arg) stage_argmax<TE>(sp, eb, ee, v0, ap);
      else if (kVec) stage_softmax(sp, vb, ve, kpv, ap);
      else stage_softmax_masked<TE>(sp, eb, ee, kpv, -INFINITY, ap);
      if (load_q) {
        if (q_arg) stage_argmax<TE>(sq, eb, ee, v0, aq);
        else if (kVec) stage_softmax(sq, vb, ve, kqv, aq);
        else stage_softmax_masked<TE>(sq, eb, ee, kqv, -INFINITY, aq);
      }
    }
    if (kVec && tid == 0) {  // the ragged tail that the bulk copies did not cover
      for (int e = nvec * PV; e < len; ++e) {
        if (p_arg) acc_scalar_argmax(ap, to_f32(sp[e]), v0 + e);
        else acc_scalar_softmax(ap, to_f32(sp[e]), kpv);
        if (load_q) {
          if (q_arg) acc_scalar_argmax(aq, to_f32(sq[e]), v0 + e);
          else acc_scalar_softmax(aq, to_f32(sq[e]), kqv);
        }
      }
    }
  } else {
    if (kVec)
      for (int s = 0; s < kStages; ++s)
        if (!mbar_wait_bounded(&ctl.bar[s], 0)) tflag = 4;
    __syncthreads();
    float tp, tq;
    TopkScratch &tk = *reinterpret_cast<TopkScratch *>(smem_raw + P.hist_off);
    topk_thresholds<TE>(sp, sq, len, topk_p, topk_q, kp_raw, kq_raw, ctl, tk, cluster, C, tp, tq);
    if (topk_p) thr_p = tp;
    if (topk_q) thr_q = tq;
    if (p_arg) stage_argmax<TE>(sp, 0, len, v0, ap);
    else stage_softmax_masked<TE>(sp, 0, len, kpv, thr_p, ap);
    if (load_q) {
      if (q_arg) stage_argmax<TE>(sq, 0, len, v0, aq);
      else stage_softmax_masked<TE>(sq, 0, len, kqv, thr_q, aq);
    }
  }
  ap.fl |= tflag;
  aq.fl |= tflag;

  // CTA partials
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    if (row == 1 && !load_q) break;
    RowAcc &a = row == 0 ? ap : aq;
    const bool arg = row == 0 ? p_arg : q_arg;
    Partial pt;
    if (arg) {
      block_argmax(a.bv, a.bi, a.fl, ctl.rs);
      pt.m = 0.f;
      pt.S = 0.f;
      pt.av = a.bv;
      pt.ai = a.bi;
    } else {
      block_online(a.m, a.S, a.fl, row == 0 ? kpv : kqv, ctl.rs);
      pt.m = a.m;
      pt.S = a.S;
      pt.av = 0.f;
      pt.ai = 0;
    }
    pt.flags = a.fl;
    if (tid == 0) ctl.part[row] = pt;
  }
  cluster_sync_all();
  // merge across the cluster (warp 0, lane r reads rank r)
  if (warp == 0) {
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (row == 1 && !load_q) break;
      const bool arg = row == 0 ? p_arg : q_arg;
      const float kk = row == 0 ? kpv : kqv;
      Partial o;
      if (lane < C) {
        o = cluster.map_shared_rank(&ctl.part[row], lane)[0];
      } else {
        o.m = -INFINITY;
        o.S = 0.f;
        o.av = -INFINITY;
        o.ai = INT_MAX;
        o.flags = 0;
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
  __syncthreads();

  // ---- 2b. top-p / min-p: a further threshold from the merged statistics,
  // then the statistics again over the entries it keeps.  The decision is the
  // same in every CTA of the cluster (per-sequence parameters and merged
  // statistics).
  {
    const float topp_v[2] = {P.pp ? __ldg(P.pp + seq) : 1.f, P.pq ? __ldg(P.pq + seq) : 1.f};
    const float minp_v[2] = {P.mp ? __ldg(P.mp + seq) : 0.f, P.mq ? __ldg(P.mq + seq) : 0.f};
    const float Tv[2] = {Tp, Tq};
    bool filt[2], do_topp[2];
    float cut[2] = {thr_p, thr_q}, mm[2], kk2[2] = {kpv, kqv}, nthr[2] = {thr_p, thr_q};
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      const bool sampled = row == 0 ? !p_arg : (load_q && !q_arg);
      const Partial o = ctl.merged[row];
      const bool finite = o.m > -INFINITY && o.m < INFINITY && !(o.flags & 3);
      filt[row] = sampled && finite && (topp_v[row] < 1.f || minp_v[row] > 0.f);
      do_topp[row] = filt[row] && topp_v[row] < 1.f;
      mm[row] = o.m;
      if (filt[row] && minp_v[row] > 0.f)
        nthr[row] = fmaxf(nthr[row], o.m + Tv[row] * logf(fminf(minp_v[row], 1.f)));
    }
    if (filt[0] || filt[1]) {
      if (do_topp[0] || do_topp[1]) {
        MassScratch &ms = *reinterpret_cast<MassScratch *>(smem_raw + P.mass_off);
        float tt[2];
        const float tpv[2] = {fmaxf(topp_v[0], 0.f), fmaxf(topp_v[1], 0.f)};
        // the histograms only over the entries min-p keeps (nthr)
        topp_thresholds<TE>(sp, sq, len, do_topp[0], do_topp[1], cut, nthr, mm, kk2, tpv, ctl,
                            ms, cluster, C, tt);
#pragma unroll
        for (int row = 0; row < 2; ++row)
          if (do_topp[row]) nthr[row] = fmaxf(nthr[row], tt[row]);
      }
      thr_p = nthr[0];
      thr_q = nthr[1];
      // every CTA has read the first round's partials before they are rewritten
      cluster_sync_all();
#pragma unroll
      for (int row = 0; row < 2; ++row) {
        if (!filt[row]) continue;
        RowAcc a;
        acc_init(a);
        stage_softmax_masked<TE>(row == 0 ? sp : sq, 0, len, kk2[row], nthr[row], a);
        block_online(a.m, a.S, a.fl, kk2[row], ctl.rs);
        Partial pt;
        pt.m = a.m;
        pt.S = a.S;
        pt.av = 0.f;
        pt.ai = 0;
        pt.flags = a.fl | ctl.merged[row].flags;
        if (tid == 0) ctl.part[row] = pt;
      }
      cluster_sync_all();
      if (warp == 0) {
#pragma unroll
        for (int row = 0; row < 2; ++row) {
          if (!filt[row]) continue;
          Partial o;
          if (lane < C) {
            o = cluster.map_shared_rank(&ctl.part[row], lane)[0];
          } else {
            o.m = -INFINITY;
            o.S = 0.f;
            o.av = -INFINITY;
            o.ai = INT_MAX;
            o.flags = 0;
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) {
            const float m2 = __shfl_xor_sync(0xFFFFFFFFu, o.m, off);
            const float S2 = __shfl_xor_sync(0xFFFFFFFFu, o.S, off);
            o.flags |= __shfl_xor_sync(0xFFFFFFFFu, o.flags, off);
            online_merge(o.m, o.S, m2, S2, kk2[row]);
          }
          if (lane == 0) ctl.merged[row] = o;
        }
      }
      __syncthreads();
    }
  }

  RowDesc dp, dq;
  bool need_fallback[2] = {false, false};
  uint32_t tmo = 0u;
#pragma unroll
  for (int row = 0; row < 2; ++row) {
    RowDesc d;
    d.m = 0.f;
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
    const Partial o = ctl.merged[row];
    if (o.flags & 4) tmo = SPEC_FLAG_TIMEOUT;
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
        need_fallback[row] = true;
        d.onehot = 1;
        d.flags = SPEC_FLAG_NONFINITE;
      }
    }
    if (row == 0) dp = d; else dq = d;
  }

  // finite-argmax fallback for non-finite sampling rows (rare)
  if (need_fallback[0] || need_fallback[1]) {
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (!need_fallback[row]) continue;
      RowAcc a;
      acc_init(a);
      stage_argmax<TE>(row == 0 ? sp : sq, 0, len, v0, a);
      block_argmax(a.bv, a.bi, a.fl, ctl.rs);
      Partial pt;
      pt.m = pt.S = 0.f;
      pt.av = a.bv;
      pt.ai = a.bi;
      pt.flags = 0;
      if (tid == 0) ctl.amax[row] = pt;
    }
    cluster_sync_all();
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

  // ---- 3. local walk over the children
  uint32_t uflags = dp.flags | tmo;
  int next = -1, token = -1;
  int residual = 0;
  float c = 0.f, Wcur = 0.f;
  int n_res = 0;
  bool have_parts = false;
  int xround = 0;
  int kind = 0;
  float total = 0.f;
  bool draw = false;
  if (dp.onehot) {
    for (; child >= 0; child = next_child(P, seq, node, child, ctl.rs)) {
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
    if (has_children) uflags |= dq.flags;
    bool first = true;
    for (; child >= 0; child = next_child(P, seq, node, child, ctl.rs)) {
      if (tid == 0) {
        const int x = child_token(P, seq, node, child);
        const int keypos = P.mode == kModeChain ? node : child;
        const float u = unit_uniform(P, seq, keypos, 0);
        int verdict = 0;  // 0 reject, 1 accept, 2 bad token, 3 zero q
        if (x < 0 || x >= V) {
          verdict = 2;
        } else {
          float zpx, zqx;
          if (first) {
            zpx = pre_zp;
            zqx = pre_zq;
          } else {
            zpx = to_f32(gp_row[x]);
            zqx = dq.onehot ? 0.f : to_f32(gq_row[x]);
          }
          const float qx = prob(dq, zqx, x);
          if (!(qx > 0.f)) {
            verdict = 3;
          } else {
            const float px =
                residual ? weight(dp, dq, 1, c, zpx, zqx, x) / Wcur : prob(dp, zpx, x);
            verdict = u < fminf(1.f, px / qx) ? 1 : 0;
          }
        }
        ctl.decision = verdict;
      }
      __syncthreads();
      const int verdict = ctl.decision;
      __syncthreads();
      first = false;
      if (verdict == 2) uflags |= SPEC_FLAG_BAD_TOKEN;
      if (verdict == 3) uflags |= SPEC_FLAG_ZERO_Q;
      if (verdict == 1) {
        next = child;
        break;
      }
      const float cn = residual ? c + Wcur : 1.f;
      const float W = cluster_total<TE>(dp, dq, 1, cn, sp, sq, v0, len, ctl, cluster, C, xround);
      if (W > 0.f) {
        residual = 1;
        c = cn;
        Wcur = W;
        ++n_res;
        have_parts = true;
      } else {
        uflags |= SPEC_FLAG_DEGENERATE_RESIDUAL;
        have_parts = false;  // ctl.parts now holds the rejected candidate's totals
      }
    }
    if (next < 0) {
      // ---- 4. inverse-CDF draw over the cluster: choose the owning CTA
      float Z;
      if (have_parts) {
        Z = Wcur;
      } else {
        Z = cluster_total<TE>(dp, dq, residual, residual ? c : 0.f, sp, sq, v0, len, ctl,
                              cluster, C, xround);
      }
      if (tid == 0) {
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
        ctl.owner = owner;
        ctl.trel = trel;
      }
      __syncthreads();
      draw = true;
      kind = has_children ? 2 : 0;
      total = Z;
    }
  }
  // A bounded wait that gave up may leave a copy in flight: wait again (also
  // bounded) before this CTA can leave.
  if (kVec && tflag)
    for (int s = 0; s < kStages; ++s) mbar_wait_bounded(&ctl.bar[s], 0);
  // Every DSMEM read of this unit is done: release the cluster; the publishing
  // CTA carries on while the others leave.
  cluster_arrive();
  const int owner = draw ? ctl.owner : 0;
  if (rank == owner) {
    if (draw) token = cta_search<TE>(dp, dq, residual, c, sp, sq, v0, len, ctl.trel, ctl);

    // ---- 5. publish this unit's outcome; the last unit of the sequence stitches
    if (tid == 0) {
      UnitOut o;
      o.next = next;
      o.token = token;
      o.flags = uflags;
      o.near = draw && ctl.margin < kRefineGuard * (1.f + (residual ? c : 0.f)) ? 1 : 0;
      P.outs[unit] = o;
      UnitStats st;
      st.p = dp;
      st.q = dq;
      st.c = residual ? c : 0.f;
      st.total = total;
      st.kind = kind;
      st.node = node;
      st.n_res = residual ? n_res : 0;
      st.pad = 0;
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
            queue_refine(P, seq, ubase + j, j, __ldcg(&P.outs[ubase + j].near));
          }
        }
      } else {
        // validate the tree: links, then depth by pointer jumping
        const int N = P.ups;
        const int32_t *par = P.parent + ubase;
        int *anc = reinterpret_cast<int *>(smem_raw + P.data_off);
        int *dep = anc + N;
        uint32_t bad = 0u;
        for (int n = tid; n < N; n += kThreads) {
          const int a = __ldg(par + n);
          if (n == 0 ? a != -1 : !(a >= 0 && a < n)) bad = 1u;
          anc[n] = n == 0 ? 0 : a;
          dep[n] = n == 0 ? 0 : 1;
        }
        bad = warp_or(bad);
        if (lane == 0) ctl.rs.red_u[warp] = bad;
        __syncthreads();
        bad = 0u;
        for (int w = 0; w < kWarps; ++w) bad |= ctl.rs.red_u[w];
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
          if (lane == 0) ctl.rs.red_u[warp] = deep;
          __syncthreads();
          deep = 0u;
          for (int w = 0; w < kWarps; ++w) deep |= ctl.rs.red_u[w];
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
          queue_refine(P, seq, ubase + cur, k, __ldcg(&P.outs[ubase + cur].near));
        }
        if (tid == 0) P.counters[seq] = 0u;
      }
    }
  }
  cluster_wait();
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
  // a sequence without a final unit (invalid tree, or a wait that gave up)
  // has no residual; an index outside the sequence's units is treated alike
  if (u < 0 || u >= P.n_units || u / P.ups != seq) {
    for (int v = vbeg + threadIdx.x; v < min(V, vbeg + kThreads * 8); v += kThreads) o[v] = 0.f;
    return;
  }
  const UnitStats st = P.stats[u];
  const int node = st.node;
  const int s2 = u / P.ups;
  if (node < 0 || node >= P.ups) {
    for (int v = vbeg + threadIdx.x; v < min(V, vbeg + kThreads * 8); v += kThreads) o[v] = 0.f;
    return;
  }
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
