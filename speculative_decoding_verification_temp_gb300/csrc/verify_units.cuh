// Fused verification kernel: one thread-block cluster per "unit".
//
// A unit is one node of the verification walk: a target row p_n, the draft
// row q_n its children were drawn from, and its children's draft tokens.  A
// chain of gamma drafts is the tree whose node i (0..gamma) has the single
// child i+1 carrying draft token x_i; node gamma is the bonus position.
//
// The outcome of the walk at a node depends only on that node's own rows,
// its children's tokens and its uniforms, so every node is resolved
// independently and in parallel ("local outcome": which child is accepted,
// or which token is drawn when none is), and the path from the root is
// stitched afterwards by the last cluster of each sequence/tree to finish.
// Each logit row is read from HBM exactly once; the row pair of a node stays
// resident in the shared memory of its cluster for every later pass
// (top-k selection, residual sums, the inverse-CDF draw).
//
// Steps inside a unit (all CTAs of the cluster run the same control flow):
//   1. load this CTA's vocabulary slice of p_n (and q_n if it has children
//      and p_n is not one-hot) into shared memory with 128-bit loads;
//   2. top-k threshold by a cluster-wide radix select over shared memory;
//   3. one pass of online max / sum of 2^((z - m) log2(e) / T) per row
//      (argmax for temperature 0), merged across the cluster through DSMEM;
//   4. the local walk: each child in ascending id gets u < min(1, p(x)/q(x));
//      on rejection p becomes norm([p - c q]_+) with c_1 = 1,
//      c_{s+1} = c_s + W_s (the closed form of repeated residuals), whose sum
//      W is reduced over the cluster;
//   5. when no child is accepted: inverse-CDF draw over the cluster: per-CTA
//      totals pick the CTA, per-warp totals the warp, a warp scan the lane;
//   6. the last unit of a sequence stitches the path (warp ballot on the
//      first rejection for chains, a walk from the root for trees).
#pragma once

#include "common.cuh"

namespace sv {

enum { kModeChain = 0, kModeTree = 1 };

// Distribution of one row after its policy.
struct RowDesc {
  int onehot;  // 1: all mass on index a
  int a;
  float k;     // log2(e) / T
  float nmk;   // -max * k
  float invS;  // 1 / sum
  float thr;   // top-k threshold (-inf: none)
  uint32_t flags;
  int pad;
};

// What a unit's final draw was taken from (read by the residual-output kernel).
struct UnitStats {
  RowDesc p, q;
  float c;      // residual multiplier (0: the draw was from p itself)
  float total;  // sum of the draw weights
  int kind;     // 0: no draw (a child was accepted) or bonus draw, 1: one-hot, 2: weights
  int node;
};

struct UnitOut {
  int next;   // accepted child node id, -1 when the unit drew `token`
  int token;
  uint32_t flags;
  int pad;
};

struct Params {
  const void *target;
  long long ld_t;
  const void *draft;
  long long ld_d;
  int V;
  int mode;
  int nseq;
  int ups;  // units per sequence: gamma + 1 (chain) or N (tree)
  int gamma;
  int max_depth;
  const int32_t *tokens;
  const int32_t *parent;
  const float *Tp;
  const float *Tq;
  const int32_t *kp;
  const int32_t *kq;
  unsigned long long seed;
  const float *uov;
  int32_t *out_num;
  int32_t *out_path;
  int32_t *out_tokens;
  uint32_t *out_flags;
  uint32_t *counters;
  UnitOut *outs;
  UnitStats *stats;
  int32_t *final_unit;
  int slice;      // vocabulary entries per CTA (multiple of 8)
  int cluster;    // CTAs per cluster
  int ctl_bytes;  // offset of the data slices in dynamic shared memory
};

struct __align__(16) Partial {
  float m, S, av;
  int ai;
  int flags;  // bit 0: NaN seen, bit 1: +inf seen
  int pad[3];
};

struct __align__(16) Ctl {
  Partial part[2];
  Partial amax[2];
  float wx[2][4];
  int hist[2][2][256];
  int ghist[2][256];
  uint32_t prefix[2];
  int kk[2];
  int child;
  int token;      // written by the owner CTA of a draw into rank 0
  int token_local;
  int owner_warp;
  float owner_t;
  int is_last;
  float parts[kMaxCluster];
  float red_f[2][kWarps];
  int red_i[2][kWarps];
  uint32_t red_u[kWarps];
};

}  // namespace sv
