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
//   1. thread 0 issues bulk asynchronous copies (TMA, cp.async.bulk) of this
//      CTA's vocabulary slice of p_n (and of q_n when the node has children
//      and p_n is not one-hot) in four stages, each completing on its own
//      mbarrier, so the whole slice is in flight at once;
//   2. as each stage lands, every thread folds its part into a running
//      max / sum of 2^((z - m) log2(e) / T) (argmax for temperature 0); the
//      per-CTA partials are merged across the cluster through DSMEM;
//      (rows with top-k first wait for the whole slice and run a cluster-wide
//      radix select for the k-th largest logit);
//   3. the local walk: each child in ascending id is accepted iff
//      u < min(1, p(x)/q(x)), with z(x) read from global memory; on rejection
//      p becomes norm([p - c q]_+) with c_1 = 1, c_{s+1} = c_s + W_s (the
//      closed form of repeated residuals), W reduced over the cluster;
//   4. when no child is accepted: inverse-CDF draw over the cluster: per-CTA
//      totals pick the CTA, per-warp totals the warp, a warp scan the lane;
//   5. one CTA publishes the unit's outcome; the last unit of a sequence to
//      publish stitches the path (warp ballot on the first rejection for
//      chains, a walk from the root for trees).
#pragma once

#include "common.cuh"

namespace sv {

enum { kModeChain = 0, kModeTree = 1 };
constexpr int kStages = 4;

// Distribution of one row after its policy.
struct RowDesc {
  int onehot;  // 1: all mass on index a
  int a;
  float k;     // log2(e) / T
  float nmk;   // -max * k
  float invS;  // 1 / sum
  float thr;   // top-k threshold (-inf: none)
  uint32_t flags;
  float m;     // row maximum (the precise redraw recomputes the weights from it)
};

// What a unit's final draw was taken from (read by the residual-output kernel).
struct UnitStats {
  RowDesc p, q;
  float c;      // residual multiplier (0: the draw was from p itself)
  float total;  // sum of the draw weights
  int kind;     // 0: no draw (a child was accepted) or bonus draw, 1: one-hot, 2: weights
  int node;
  int n_res;    // residual rounds that set the multiplier: c = c_{n_res} (0: p itself)
  int pad;
};

struct UnitOut {
  int next;   // accepted child node id, -1 when the unit drew `token`
  int token;
  uint32_t flags;
  int near;   // 1: the draw fell within the refine guard of a CDF boundary
};

// A final draw whose single-precision running sum came within this distance
// (in probability units, times 1 + c for a residual [p - c q]_+) of a CDF
// boundary is redrawn in double-float arithmetic by the refine kernel.
constexpr float kRefineGuard = 4e-6f;

// The precise redraw runs on at most this many CTAs.
constexpr int kRefineMaxGrid = 1024;

// 64-bit records the chain rows kernel leaves per 32 KB chunk (one per
// consumer warp).
constexpr int kChainRecordsPerChunk = 8;

// Largest tree (nodes) the tree walk over the rows stream takes; larger trees
// go to the streaming or resident kernel.
constexpr int kWalkMaxNodes = 256;

// One work unit of the precise redraw (a slice of one queued draw's
// vocabulary): its partial sums, published for the other units of the draw.
// A chain's final draw: the decision the chain draw kernel's CTAs share, and
// the description a queued precise redraw reads.
struct __align__(16) PassSeq {
  RowDesc dp, dq;  // the draw distribution: [p - q]_+ (residual) or p
  float u;         // draw uniform
  float W;         // single-precision total of the draw weights
  int residual;
  int j;           // draw position
  uint32_t flags;
  int kind;        // 0: bonus draw, 1: one-hot, 2: residual draw (UnitStats::kind)
  int draw;        // 1: weight jobs run the draw; 0: the token needed no draw
};

struct __align__(16) RefinePart {
  double a, b;           // shares of the softmax normalisers S_p, S_q
  double rw;             // share of a residual round's total W_s
  double w;              // share of the final draw's total
  double warp[kWarps];   // per-warp totals of the final weights
  int wlast[kWarps];     // per-warp last entry with positive weight (-1: none)
  int last;              // the unit's last entry with positive weight
  int pad[3];
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
  const float *pp;  // top-p per sequence (NULL: none)
  const float *pq;
  const float *mp;  // min-p per sequence (NULL: none)
  const float *mq;
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
  int data_off;   // byte offset of the data slices in dynamic shared memory
  int hist_off;   // byte offset of the top-k histograms (0: no top-k in this launch)
  int mass_off;   // byte offset of the top-p mass histograms (0: no top-p in this launch)
  long long first_wait;  // cycles the chain rows kernel's first wait on a chunk may take
  // streaming (persistent) kernel only
  const int32_t *first_child;  // [T*N] first child of each tree node, -1 for leaves
  int n_units;
  int ring;                       // ring slots per CTA
  int slot_bytes;                 // bytes per ring slot
  int chunks;                     // ring chunks per row slice
  int slice_blocks;               // draw blocks per slice (chunks * 16 + 1)
  struct SlicePartial *partials;  // [n_units][slices][2]
  struct DrawState *dstate;       // [n_units]
  float *wpart;                   // [n_units][slices] slice totals of the round
  float *wblk;                    // [n_units][slices][slice_blocks] block totals
  uint32_t *unit_done;            // [n_units] stats slices finished
  uint32_t *w_done;               // [n_units] weight slices finished in the round
  int4 *wq;                       // weight-task queue: (unit, slice, round, epoch)
  uint32_t *wq_ctr;               // [0] head, [1] tail, [2] units completed
  uint32_t epoch;                 // tags this call's queue entries
  int wq_cap;
  // precise redraw of final draws near a CDF boundary
  int4 *refine;                   // [nseq] (seq, unit, output position, 0)
  uint32_t *refine_ctr;           // entries in `refine`
  RefinePart *rpart;              // [max(kRefineMaxGrid, nseq)] work-unit partials
  double *rc;                     // [nseq] residual multiplier of each queued draw
  uint32_t *rbar;                 // grid-barrier arrivals of the redraw kernel
  // streaming chain path (rows kernel, draw kernel, precise kernel)
  unsigned long long *srec;       // [rows][chunks][8] per-warp records of the rows kernel
  float4 *trec;                   // typical acceptance: [rows][chunks][8] (max, S1, S2, index)
  uint32_t *err;                  // bit 0: a bounded wait gave up
  int chunk_elems;                // entries per chunk
  int cpr;                        // chunks per row
  int steps;                      // draw search steps per row (256 entries each)
  void *bmax;                     // [rows][nblk] the rows' 512-entry block maxima (element
                                  //   type; NULL: no row filter in the call)
  float2 *frec;                   // [rows] filtered rows: (threshold, kept normaliser S)
  int nblk;                       // 512-entry blocks per row
  int walk_buf;                   // tree walk: bytes of a CTA's staging buffer
  unsigned long long *pseqw;      // [nseq] PassSeq of each queued precise redraw
  int *near_list;                 // [nseq] sequence + 1 of each queued precise redraw
  uint32_t *pctr;                 // [0] precise redraws queued (cleared by every call)
};



struct __align__(16) Partial {
  float m, S, av;
  int ai;
  int flags;  // bit 0: NaN seen, bit 1: +inf seen, bit 2: bounded wait timed out
  int pad[3];
};

// Scratch of the CTA-wide reductions and of the child scan.
struct RedScratch {
  float red_f[2][kWarps];
  int red_i[2][kWarps];
  uint32_t red_u[kWarps];
  int child;
};

struct TopkScratch {
  int hist[2][2][256];
  int ghist[2][256];
};

// Mass histograms of the top-p select (fixed point, see topp_thresholds).
struct MassScratch {
  unsigned long long hist[2][2][256];
  unsigned long long ghist[2][256];
  unsigned long long remaining[2];
  unsigned long long wtot[kWarps][2];  // round 0: per-warp total masses
  unsigned long long ctot[2];          // this CTA's total masses
  unsigned long long gtot[2];          // the cluster's total masses
  int below[2];                        // the top-p boundary lies below hcut
};

struct __align__(16) Ctl {
  unsigned long long bar[kStages];
  Partial part[2];
  Partial amax[2];
  Partial merged[2];
  float wx[2][4];
  float parts[kMaxCluster];
  uint32_t prefix[2];
  int kk[2];
  int token_local;
  int owner_warp;
  float owner_t;
  int is_last;
  int decision;  // broadcast of thread 0's per-child verdict
  int owner;
  float trel;
  float margin;  // distance of the draw from the nearer CDF boundary
  RedScratch rs;
};

// ---------------------------------------------------------------------------
// streaming kernel state
// ---------------------------------------------------------------------------

constexpr int kMaxRing = 8;
constexpr int kBlocksPerChunk = 16;  // draw-weight blocks per ring chunk (search granularity)
constexpr int kMaxSliceBlocks = 2 * kBlocksPerChunk + 1;  // two chunks and the ragged tail

enum { kTaskStats = 0, kTaskWeights = 1, kTaskEnd = 2 };

// One CTA's statistics of its slice of one row, published for the unit's
// deciding CTA.
struct __align__(16) SlicePartial {
  float m, S, av;
  int ai;
  int flags;  // bit 0: NaN seen, bit 1: +inf seen, bit 2: bounded wait timed out
  int pad[3];
};

// A unit's draw state between weight rounds (workspace, one per unit).
struct __align__(16) DrawState {
  RowDesc dp, dq;
  float c;       // multiplier of the round in flight (0: the weights are p itself)
  float c_cur;   // multiplier of the distribution the node holds (0: p)
  float W_cur;   // its total (valid when c_cur > 0)
  int child;     // the last child tested
  uint32_t flags;
  int round;
  int blocks_c_valid;  // 1 when the stored block totals belong to the held distribution
  int n_res;           // residual rounds that set c_cur
};

// What the producer warp tells the compute threads about a task.
struct __align__(16) TaskInfo {
  int type, unit, slice, round;
  int bits;  // stats: 1 p_arg, 2 q_arg, 4 tp_bad, 8 tq_bad, 16 load_q, 32 has_children
  float kp, kq;
  float c;   // weights: round multiplier
  RowDesc dp, dq;
};

struct __align__(16) Ctl3 {
  unsigned long long full[kMaxRing];
  unsigned long long empty[kMaxRing];
  TaskInfo tinfo[kMaxRing];
  float btot[kMaxSliceBlocks + 15];
  Partial merged[2];
  DrawState ds_share;  // draw state handed from thread 0 to warp 0
  int decision;
  int is_last;
  int token;
  float trel;
  RedScratch rs;
};

}  // namespace sv
